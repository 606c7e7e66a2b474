"""Full-size parity on the 480p-shaped layer (40 heads, 8 chunks of 4,680 tokens = 36 full 128-token
tiles + a ragged 72-row tile; 4,680 Queries = 9 items of 512 rows + a 72-row short item) in the
launch configuration of the benchmark: the stream of the 480p layer itself, one sampled layer (the
last, layer 39) of the 40-layer model built from that layer shape, and the extremes of the ablation
sweep on the same shapes.  The oracle recomputes sampled outputs one by one from the GPU's upstream
state, the ragged tile's rows and the short attention item's rows always among them."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import synth  # noqa: E402
from fullsize import (check_attention, check_decoder, check_kmeans, check_packing,  # noqa: E402
                      check_statistics, stream_layer)

W = synth.P480
N = W.chunk_tokens          # 4,680
NQ = W.nq_attend            # 4,680


def packing_rows(n_random: int, seed: int):
    rng = np.random.default_rng(seed)
    tail = np.r_[4606:4612, 4640, 4677:N]  # around the last full tile and the ragged 72-row tile
    return np.unique(np.r_[0, 127, 128, tail, rng.choice(N, n_random, replace=False)])


def attention_rows(n_random: int, seed: int):
    rng = np.random.default_rng(seed)
    # row 0, tile and item boundaries, and rows of the 72-row short item (4,608..4,679)
    return np.unique(np.r_[0, 255, 256, 511, 512, 4607, 4608, 4650, NQ - 1, rng.choice(NQ, n_random, replace=False)])


@pytest.fixture(scope="module", params=[0, 39], ids=["layer0", "model_layer39"])
def run(request):
    import __graft_entry__
    __graft_entry__.build_library()
    return stream_layer(W, layer=request.param)


def test_statistics(run):
    check_statistics(run, (0, 39))


def test_kmeans_objective(run):
    check_kmeans(run, 11, "k")
    check_kmeans(run, 30, "v")


def test_packing_sampled_tokens_with_ragged_tile(run):
    ties = check_packing(run, (0, 17, 39), packing_rows(120, 2))
    print(f"ties (score, candidate boundary, value): {ties.tolist()}")


def test_decoder(run):
    check_decoder(run, 5)
    check_decoder(run, 36, chunk=0)  # the cold-start chunk (no PSAC)


def test_attention_rows_incl_short_item(run):
    worst = check_attention(run, (0, 39), attention_rows(6, 3))
    print(f"attention max error {worst:.2e} x RMS(O)")


@pytest.mark.parametrize("C,M,r", [(64, 1, 0), (1024, 16, 16)], ids=["C64_M1_r0", "C1024_M16_r16"])
def test_ablation_extremes_at_480p(C, M, r):
    """The two ends of the M x r x C sweep streamed at full 480p size: packing, codebook and attention
    parity on sampled heads, tokens and rows."""
    import __graft_entry__
    __graft_entry__.build_library()
    run = stream_layer(W, layer=0, n_centroids=C, top_m=M, rank=r, kmeans_iters=10)
    check_kmeans(run, 3, "k")
    check_packing(run, (2, 38), packing_rows(40, 5))
    check_decoder(run, 21)
    check_attention(run, (1,), attention_rows(2, 7))
