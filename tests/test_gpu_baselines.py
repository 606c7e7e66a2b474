"""GPU-vs-oracle parity of the comparison baselines (include/qwm_baselines.h), through the C ABI.

  * KIVI-style INT2 (per-channel Keys over 32-token groups, per-token Values over 32-channel groups):
    codes, fp16 steps and offsets bit-exact; the decode bit-exact (m + s q is one rounding on both sides);
  * QVG two-stage progressive residual quantisation: stage indices as the QuantWM parity bar (exact
    except near-ties), the stage residual bit-exact given the indices, the second stage's codes bit-exact
    given its indices, the fused two-stage decode within one bf16 step (plus the fp32 error of a sum
    that cancels).
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import oracle  # noqa: E402
import synth  # noqa: E402
from helpers import bf16_ulp_close, chunk_head, from_u16, to_u16  # noqa: E402

D = 128
TIE = 1e-5


@pytest.fixture(scope="module")
def q():
    import __graft_entry__
    __graft_entry__.build_library()
    import bit_kv_cache_qsac_gb300 as qq
    assert torch.cuda.is_available()
    return qq


def _bf(a):
    return from_u16(a, torch.bfloat16)


def _f64(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


@pytest.mark.parametrize("n", [1000, 64, 7])
def test_kivi_quantize_and_decode_bit_exact(q, n):
    H = 2
    k = synth.keys(synth.TINY)[:H, :n]; v = synth.values(synth.TINY)[:H, :n]
    ctx = q.Context(heads=H)
    ch = q.KiviChunk.empty(ctx, n)
    q.qwm_kivi_quantize(ctx, _bf(k), _bf(v), n, ch)
    kh = torch.empty(H, n, D, dtype=torch.bfloat16, device="cuda"); vh = torch.empty_like(kh)
    q.qwm_kivi_dequantize(ctx, ch, kh, vh)
    assert q.qwm_sync_status(ctx) == 0
    for h in range(H):
        o = oracle.kivi_quantize_head(k[h], v[h], 32)
        for name in ("k_codes", "v_codes"):
            assert np.array_equal(getattr(ch, name)[h].cpu().numpy(), o[name]), name
        for name in ("k_scale", "k_min", "v_scale", "v_min"):
            assert np.array_equal(to_u16(getattr(ch, name)[h]), o[name]), name
        k64, v64 = oracle.kivi_dequantize_head(o, 32)
        rne = np.vectorize(oracle.bf16_rne)
        assert np.array_equal(to_u16(kh[h]), rne(k64).astype(np.uint16))
        assert np.array_equal(to_u16(vh[h]), rne(v64).astype(np.uint16))


def _stage(q, ctx, K, V, n):
    """One nearest-centroid stage on the GPU: k-means codebooks, then the quantiser with a single
    candidate, no weights and no PSAC (exactly nearest-centroid assignment)."""
    ch = q.Chunk.empty(ctx, n)
    q.qwm_fit_centroids(ctx, K, n, None, ch.cent_k)
    q.qwm_fit_centroids(ctx, V, n, None, ch.cent_v)
    q.qwm_quantize_kv(ctx, K, V, n, None, None, ch)
    return ch


def test_prq_two_stage(q):
    H, n, C = 2, 1000, 64
    w_ = synth.TINY
    k = synth.keys(w_)[:H, :n]; v = synth.values(w_)[:H, :n]
    ctx = q.Context(heads=H, n_centroids=C, top_m=1, rank=0)
    K, V = _bf(k), _bf(v)
    ch1 = _stage(q, ctx, K, V, n)
    r1k = torch.empty_like(K); r1v = torch.empty_like(V)
    q.qwm_prq_residual(ctx, K, n, ch1.cent_k, ch1.k_idx, r1k)
    q.qwm_prq_residual(ctx, V, n, ch1.cent_v, ch1.v_idx, r1v)
    ch2 = _stage(q, ctx, r1k, r1v, n)
    kh = torch.empty(H, n, D, dtype=torch.bfloat16, device="cuda"); vh = torch.empty_like(kh)
    q.qwm_prq_dequantize(ctx, ch2, ch1.cent_k, ch1.k_idx, ch1.cent_v, ch1.v_idx, kh, vh)
    assert q.qwm_sync_status(ctx) == 0
    for h in range(H):
        c1k, c1v = to_u16(ch1.cent_k[h]), to_u16(ch1.cent_v[h])
        i1k = ch1.k_idx[h].cpu().numpy().astype(np.int32); i1v = ch1.v_idx[h].cpu().numpy().astype(np.int32)
        # stage 1: nearest centroid (ties within a relative 1e-5 may go either way)
        o1 = oracle.quantize_head(k[h], v[h], c1k, c1v, None, None, top_m=1, rank=0)
        for gi, oi, dist in ((i1k, o1["idx_k"], o1["dq_edge"]), (i1v, o1["idx_v"], o1["vdist2"])):
            tie = np.abs(dist[:, 1] - dist[:, 0]) <= TIE * np.abs(dist[:, 0])
            assert np.all((gi == oi) | tie)
        # stage residual: bit-exact given the GPU's indices
        assert np.array_equal(to_u16(r1k[h]), oracle.prq_residual(k[h], c1k, i1k))
        assert np.array_equal(to_u16(r1v[h]), oracle.prq_residual(v[h], c1v, i1v))
        # stage 2 codes given its indices
        i2k = ch2.k_idx[h].cpu().numpy().astype(np.int32); i2v = ch2.v_idx[h].cpu().numpy().astype(np.int32)
        o2 = oracle.quantize_head(to_u16(r1k[h]), to_u16(r1v[h]), to_u16(ch2.cent_k[h]), to_u16(ch2.cent_v[h]),
                                  None, None, top_m=1, rank=0, force_idx_k=i2k, force_idx_v=i2v)
        for name in ("k_codes", "v_codes"):
            assert np.array_equal(getattr(ch2, name)[h].cpu().numpy(), o2[name]), name
        for name in ("k_scale", "k_min", "v_scale", "v_min"):
            assert np.array_equal(to_u16(getattr(ch2, name)[h]), o2[name]), name
        # fused decode: mu1 + (mu2 + r_hat) against the oracle's double sum
        # (the two-stage decoder reads the stage codebooks in bf16, as QVG stores them)
        c2 = chunk_head(ch2, h)
        del c2["cent_k16"], c2["cent_v16"]
        c2["cent_k"], c2["cent_v"] = to_u16(ch2.cent_k[h]), to_u16(ch2.cent_v[h])
        _, _, k2, v2 = oracle.dequantize_head(c2)
        for got, ref2, cent1, i1, key in ((kh[h], k2, c1k, i1k, "k"), (vh[h], v2, c1v, i1v, "v")):
            ref = ref2 + _f64(cent1[i1])
            g = _f64(to_u16(got))
            mag = np.abs(_f64(cent1[i1])) + np.abs(ref2) + np.abs(_f64(c2["cent_" + key][c2["idx_" + key]]))
            assert np.all(bf16_ulp_close(to_u16(got), ref) | (np.abs(g - ref) <= 2.0 ** -20 * mag)), key
