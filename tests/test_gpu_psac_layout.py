"""PSAC rank per (chunk, head) and the per-head coefficient layout, through the C ABI, against the
oracle: the rank rule on the GPU's eigenvalues, packing with per-head ranks, the kept counts, the
dense-or-sparse choice and the sparse rows (bit-exact), and attention and decoding over a chunk in the
per-head layout (identical to the same chunk in the dense layout, and within the attention bar of the
oracle)."""
import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import oracle  # noqa: E402
import synth  # noqa: E402
from helpers import bf16_ulp_close, chunk_head, decode_term_magnitude, from_u16, psac_dense_head, to_u16  # noqa: E402

D = 128
W4 = synth.Workload("psac-4-heads", 4, heads=4, frames=6, hs=30, ws=52, frames_per_chunk=3,
                    nq_stats=1024, nq_attend=300)


@pytest.fixture(scope="module")
def q():
    import __graft_entry__
    __graft_entry__.build_library()
    import bit_kv_cache_qsac_gb300 as qq
    return qq


def _bf(a):
    return from_u16(a, torch.bfloat16)


def attention_close(got, ref):
    """The attention bar, max |error| <= 2e-2 x RMS(O), for heads whose outputs peak below 25 x RMS(O).
    One synthetic head of this 4-head workload peaks at ~42 x RMS(O) (a few keys dominate its
    softmax and their Values carry the x8 outlier channels); there the fp16 rounding of the decoded
    outlier values alone (one fp16 unit of ~9.5 is 0.008) exceeds that bar, whatever the layout, so
    such a head is held to 1e-3 of its peak instead (about two fp16 units)."""
    err = np.abs(got - ref).max()
    rms, peak = math.sqrt(np.mean(ref ** 2)), np.abs(ref).max()
    return err <= 2e-2 * rms if peak < 25 * rms else err <= 1e-3 * peak


def mixed_queries(t, nq, H=4):
    """Queries whose spectra differ by head (32 channels lifted by a per-head factor), so that the
    energy rule gives different ranks to different heads."""
    qs = synth.bf16_bits_to_f32(synth.queries(W4, t, nq)[:H]).astype(np.float32)
    for h in range(H):
        qs[h][:, :32] *= 1.0 + 0.5 * h
    return synth.f32_to_bf16_bits(qs)


def _stats(q, ctx, H, nq=1024, seed=0):
    S = torch.zeros(H, D, D, device="cuda"); n = torch.zeros(H, dtype=torch.int64, device="cuda")
    w = torch.empty(H, D, device="cuda"); lam = torch.empty(H, D, device="cuda")
    ur = torch.zeros(H, D, ctx.cfg.rank, dtype=torch.bfloat16, device="cuda")
    q.qwm_update_query_stats(ctx, _bf(mixed_queries(seed, nq, H)), nq, S, n, w, lam, ur)
    return w, lam, ur


@pytest.mark.parametrize("energy", [0.0, 0.3, 0.55, 0.7, 1.0])
def test_select_rank_rule(q, energy):
    H, R = 4, 16
    ctx = q.Context(heads=H, rank=R)
    _, lam, ur = _stats(q, ctx, H)
    ur0 = ur.clone()
    hr = torch.empty(H, dtype=torch.int32, device="cuda")
    q.qwm_select_rank(ctx, lam, energy, ur, hr)
    assert q.qwm_sync_status(ctx) == 0
    e32 = float(np.float32(energy))                     # the library takes the share as fp32
    for h in range(H):
        want = oracle.adaptive_rank(lam[h].cpu().numpy(), R, e32)
        r = int(hr[h])
        assert r == want, (h, r, want)
        assert torch.equal(ur[h, :, :r], ur0[h, :, :r]) and not ur[h, :, r:].float().abs().sum()


def _packed_with_ranks(q, energy=0.55, gate=0, w_override=None, u_override=None, n=1000):
    """Four heads packed with per-head ranks (and optionally the gate, weights and bases given)."""
    H, R = 4, 8
    ctx = q.Context(heads=H, rank=R, psac_gate=gate)
    w, lam, ur = _stats(q, ctx, H)
    if w_override is not None:
        w = torch.from_numpy(w_override).float().cuda().contiguous()
    if u_override is not None:
        ur = from_u16(u_override, torch.bfloat16)
    hr = torch.full((H,), R, dtype=torch.int32, device="cuda")
    if energy is not None:
        q.qwm_select_rank(ctx, lam, energy, ur, hr)
    k = synth.keys(W4)[:H, :n]; v = synth.values(W4)[:H, :n]
    ch = q.Chunk.empty(ctx, n)
    K, V = _bf(np.ascontiguousarray(k)), _bf(np.ascontiguousarray(v))
    q.qwm_fit_centroids(ctx, K, n, None, ch.cent_k)
    q.qwm_fit_centroids(ctx, V, n, None, ch.cent_v)
    ch.u_r.copy_(ur)
    dbg = dict(c_f32=torch.zeros(H, n, R, device="cuda"))
    q.qwm_quantize_kv(ctx, K, V, n, w, ch.u_r, ch, dbg)
    assert q.qwm_sync_status(ctx) == 0
    return ctx, ch, k, v, w, hr, dbg


def test_quantize_with_per_head_ranks(q):
    """Coefficients past a head's rank are zero; its first r_h are the oracle's rank-r_h packing."""
    ctx, ch, k, v, w, hr, dbg = _packed_with_ranks(q, energy=0.55)
    ranks = hr.cpu().tolist()
    print("ranks", ranks)
    for h, r in enumerate(ranks):
        cg = dbg["c_f32"][h].cpu().numpy().astype(np.float64)
        assert not np.any(cg[:, r:])
        assert not np.any(ch.c[h].cpu().numpy()[:, r:])
        if r == 0:
            assert not np.any(to_u16(ch.c_scale[h]))
            continue
        ur = to_u16(ch.u_r[h])[:, :r]
        o = oracle.quantize_head(k[h], v[h], to_u16(ch.cent_k[h]), to_u16(ch.cent_v[h]),
                                 w[h].cpu().numpy().astype(np.float64), ur, top_m=4, rank=r,
                                 force_idx_k=ch.k_idx[h].cpu().numpy().astype(np.int32),
                                 force_idx_v=ch.v_idx[h].cpu().numpy().astype(np.int32))
        scale_ = np.maximum(np.abs(o["c_real"]).max(1, keepdims=True), 1e-30)
        assert np.all(np.abs(cg[:, :r] - o["c_real"]) <= 1e-3 * scale_)
        gc8, gsc = ch.c[h].cpu().numpy()[:, :r], to_u16(ch.c_scale[h])
        for i in range(k.shape[1]):
            c8, sc = oracle.int8_encode_token(cg[i, :r].astype(np.float32))
            assert sc == gsc[i] and np.array_equal(c8, gc8[i])


def _gate_case():
    """Per-head bases against weights that are zero on channels 64..127: head 0's basis sees only
    unweighted channels (the gate drops every token), heads 1 and 2 lean on them (the gate drops
    most tokens), head 3 keeps its statistics' basis."""
    H = 4
    w = np.ones((H, D))
    w[:3, 64:] = 0.0
    U = np.zeros((H, D, 8))
    for h, a in ((0, 0.0), (1, 0.5), (2, 0.2)):
        U[h, 64 + np.arange(8) * 8, np.arange(8)] = 1.0
        U[h, np.arange(8) * 8, np.arange(8)] = a
        U[h] /= np.linalg.norm(U[h], axis=0)
    return w, U


def test_psac_pack_layout_bit_exact(q):
    w, U = _gate_case()
    _, lam, ur = _stats(q, q.Context(heads=4, rank=8), 4)
    Ub = to_u16(ur).copy()
    Ub[:3] = synth.f32_to_bf16_bits(U[:3].astype(np.float32))
    ctx, ch, k, v, wt, hr, dbg = _packed_with_ranks(q, energy=None, gate=1, w_override=w, u_override=Ub, n=1000)
    H, n = 4, 1000
    c_dense = [ch.c[h].cpu().numpy().copy() for h in range(H)]
    s_dense = [to_u16(ch.c_scale[h]).copy() for h in range(H)]
    kept_o = [int((s != 0).sum()) for s in s_dense]
    assert kept_o[0] == 0 and 0 < kept_o[1] < 0.7 * n and 0 < kept_o[2] < 0.7 * n and kept_o[3] > 0.8 * n, kept_o
    q.pack_psac_layout(ctx, ch, hr)
    assert q.qwm_sync_status(ctx) == 0
    plan_o = oracle.psac_plan(n, [8] * H, kept_o)
    for h in range(H):
        c_off, s_off, rh, sparse = ch.plan[h]
        assert (bool(sparse), rh) == (plan_o[h][0], 8)
        rows = plan_o[h][1]
        got_c = ch.c.cpu().numpy()[c_off:c_off + rows * 8].reshape(rows, 8)
        got_s = to_u16(ch.c_scale)[s_off:s_off + rows]
        if sparse:
            mask, trank, rows_o, sc_o = oracle.psac_sparse_encode(c_dense[h], s_dense[h])
            assert np.array_equal(ch.c_mask[h].cpu().numpy().view(np.uint32), mask)
            assert np.array_equal(ch.c_tile_rank[h].cpu().numpy(), trank)
            assert np.array_equal(got_c, rows_o) and np.array_equal(got_s, sc_o)
        else:
            assert np.array_equal(got_c, c_dense[h]) and np.array_equal(got_s, s_dense[h])
        cd, sd = psac_dense_head(ch, h)
        assert np.array_equal(cd, c_dense[h]) and np.array_equal(sd, s_dense[h])
    assert ch.plan[0][3] == 1 and ch.plan[1][3] == 1      # the heads whose gate drops many tokens go sparse
    dense_bytes = H * n * 10
    assert ch.c.numel() + 2 * ch.c_scale.numel() <= 0.6 * dense_bytes


def _dense_twin(q, ch):
    """The same packed chunk with its dense coefficients rebuilt from the per-head layout."""
    import copy
    tw = copy.copy(ch)
    H, n, r = ch.c_mask.shape[0], ch.n_tokens, ch.rank_eff
    c = np.zeros((H, n, r), np.int8); sc = np.zeros((H, n), np.uint16)
    for h in range(H):
        c[h], sc[h] = psac_dense_head(ch, h)
    tw.c = torch.from_numpy(c).cuda()
    tw.c_scale = torch.from_numpy(sc.view(np.int16)).cuda().view(torch.float16)
    tw.c_layout, tw.c_heads, tw.c_mask, tw.c_tile_rank, tw.plan = 0, None, None, None, None
    return tw


@pytest.mark.parametrize("case", ["ranks", "gate"])
def test_attend_and_decode_per_head_layout(q, case):
    if case == "ranks":
        ctx, ch, k, v, w, hr, _ = _packed_with_ranks(q, energy=0.55, n=777)
    else:
        wt, U = _gate_case()
        _, lam, ur = _stats(q, q.Context(heads=4, rank=8), 4)
        Ub = to_u16(ur).copy()
        Ub[:3] = synth.f32_to_bf16_bits(U[:3].astype(np.float32))
        ctx, ch, k, v, w, hr, _ = _packed_with_ranks(q, energy=0.7, gate=1, w_override=wt, u_override=Ub, n=777)
    q.pack_psac_layout(ctx, ch, hr)
    tw = _dense_twin(q, ch)
    H, nq = 4, 300
    qa = synth.queries(W4, 5, nq)[:H]
    out = torch.empty(H, nq, D, dtype=torch.float32, device="cuda")
    out2 = torch.empty_like(out)
    q.qwm_attend(ctx, _bf(qa), nq, [ch], 1 / math.sqrt(D), out)
    q.qwm_attend(ctx, _bf(qa), nq, [tw], 1 / math.sqrt(D), out2)
    assert q.qwm_sync_status(ctx) == 0
    assert torch.equal(out, out2)
    kh = torch.empty(H, ch.n_tokens, D, dtype=torch.bfloat16, device="cuda"); vh = torch.empty_like(kh)
    kh2, vh2 = torch.empty_like(kh), torch.empty_like(kh)
    q.qwm_dequantize(ctx, ch, kh, vh)
    q.qwm_dequantize(ctx, tw, kh2, vh2)
    assert q.qwm_sync_status(ctx) == 0
    assert torch.equal(kh, kh2) and torch.equal(vh, vh2)
    for h in range(H):
        c = chunk_head(ch, h)
        ref = oracle.attend_rows(qa[h], np.arange(nq), [c], 1 / math.sqrt(D))
        got = out[h].cpu().numpy().astype(np.float64)
        assert attention_close(got, ref), (h, np.abs(got - ref).max(), math.sqrt(np.mean(ref ** 2)), np.abs(ref).max())
        _, _, k64, _ = oracle.dequantize_head(c)
        g = (to_u16(kh[h]).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        slack = 2.0 ** -20 * decode_term_magnitude(c, True)
        assert (bf16_ulp_close(to_u16(kh[h]), k64) | (np.abs(g - k64) <= slack)).all()


def test_stream_with_adaptive_rank_and_per_head_layout(q):
    """A streamed layer with per-chunk, per-head ranks (energy share 0.55) and the gate: attention over
    every chunk matches the oracle, and the cache is smaller than the fixed-rank dense one."""
    from bit_kv_cache_qsac_gb300.stream import CompressedLayer
    H = 4
    ks, vs = synth.keys(W4)[:H], synth.values(W4)[:H]
    layers = []
    for adaptive in (False, True):
        ctx = q.Context(heads=H, psac_gate=1)
        lay = CompressedLayer(ctx, rank_energy=0.55 if adaptive else None)
        for t, (a, b) in enumerate([(0, 1560), (1560, 3120), (3120, 4680)]):
            if t:
                lay.fold_queries(_bf(mixed_queries(40 + t, 600, H)))
            lay.append_chunk(_bf(np.ascontiguousarray(ks[:, a:b])), _bf(np.ascontiguousarray(vs[:, a:b])))
        assert lay.check() == 0
        layers.append(lay)
    lay = layers[1]
    assert all(c.c_layout == 1 for c in lay.chunks[1:])
    assert len({r for c in lay.chunks[1:] for r in c.head_rank.tolist()}) > 1
    assert lay.nbytes() < layers[0].nbytes()
    qa = synth.queries(W4, 9, 200)[:H]
    out = lay.attend(_bf(qa))
    assert lay.check() == 0
    for h in range(H):
        ref = oracle.attend_rows(qa[h], np.arange(200), [chunk_head(c, h) for c in lay.chunks], 1 / math.sqrt(D))
        got = out[h].cpu().numpy().astype(np.float64)
        assert attention_close(got, ref), (h, np.abs(got - ref).max(), math.sqrt(np.mean(ref ** 2)))
