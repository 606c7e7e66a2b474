"""GPU-vs-oracle parity of every step of the path, called through the C ABI.

Stage-wise protocol: each GPU stage is compared with the oracle run on the GPU's own
upstream outputs (statistics -> basis -> codebooks -> packing -> attention), so that
tolerances do not compound.  Bars (from the method's definition of equivalence):
  * centroid indices: bit-exact except where the oracle's best and second-best QSAC
    score (Values: distance), or its M-th and (M+1)-th d_Q, lie within a relative 1e-5;
  * INT2 codes, packed bytes, fp16 scales and offsets: bit-exact given the index;
  * INT8 PSAC codes and scales: bit-exact given the unquantised fp32 coefficients;
    those coefficients within a relative 1e-3 of the oracle's (of the token's max |C|);
  * eigenvalues within a relative 1e-3;
  * attention output: max |error| <= 2e-2 x RMS(O);
  * decoder: within one bf16 step, or within 2^-20 x the sum of the decoded terms' magnitudes
    where that sum cancels (the decoder evaluates in fp32).
"""
import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import oracle  # noqa: E402
import synth  # noqa: E402
from helpers import bf16_ulp_close, chunk_head, decode_term_magnitude, from_u16, to_u16  # noqa: E402

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


def _f32(bits):
    return synth.bf16_bits_to_f32(bits).astype(np.float64)


# ------------------------------------------------------------------ step 1


def test_stats_weights_and_basis(q):
    w_ = synth.TINY
    H = w_.heads
    ctx = q.Context(heads=H)
    S = torch.zeros(H, D, D, device="cuda"); n = torch.zeros(H, dtype=torch.int64, device="cuda")
    w = torch.empty(H, D, device="cuda"); lam = torch.empty(H, D, device="cuda")
    ur = torch.empty(H, D, 8, dtype=torch.bfloat16, device="cuda")
    # cold start: no Queries yet
    q.qwm_update_query_stats(ctx, None, 0, S, n, w, lam, ur)
    assert q.qwm_sync_status(ctx) == 0
    assert torch.all(w == 1) and torch.all(lam == 0) and torch.all(n == 0)
    S64 = np.zeros((H, D, D)); n64 = np.zeros(H, np.int64)
    for batch, nq in enumerate((256, 100)):    # second batch: incremental, ragged size
        qb = synth.queries(w_, batch - 1, nq)
        q.qwm_update_query_stats(ctx, _bf(qb), nq, S, n, w, lam, ur)
        assert q.qwm_sync_status(ctx) == 0
        ow, olam, our, oU, _ = oracle.update_query_stats(qb, S64, n64, 8)
        assert np.array_equal(n.cpu().numpy(), n64)
        np.testing.assert_allclose(S.cpu().numpy(), S64, rtol=1e-5, atol=1e-5 * np.abs(S64).max())
        np.testing.assert_allclose(w.cpu().numpy(), ow, rtol=1e-5)
        gl = lam.cpu().numpy()
        assert np.all(np.abs(gl - olam) <= 1e-3 * np.abs(olam) + 1e-6 * np.abs(olam).max())
        gu = _f32(to_u16(ur))
        for h in range(H):
            for kk in range(8):
                u_ref = oU[h][:, kk]
                cosv = gu[h][:, kk] @ u_ref / np.linalg.norm(gu[h][:, kk])
                assert cosv > 0.999, (h, kk, cosv)            # same direction and sign convention
            # bf16 rounding of the same vector: within one bf16 step where the vectors agree closely
            assert np.mean(bf16_ulp_close(to_u16(ur[h]), oU[h][:, :8], 1.0)) > 0.95


def test_basis_rank16_eigenpairs(q):
    """Rank 16 reaches into the noise eigenvalues: every returned column is an eigenvector of M
    (residual at the bf16 rounding level), the columns are orthonormal to that level, the first 8
    match the oracle's, and all 128 eigenvalues agree."""
    w_ = synth.TINY
    H = w_.heads
    ctx = q.Context(heads=H, rank=16)
    S = torch.zeros(H, D, D, device="cuda"); n = torch.zeros(H, dtype=torch.int64, device="cuda")
    w = torch.empty(H, D, device="cuda"); lam = torch.empty(H, D, device="cuda")
    ur = torch.empty(H, D, 16, dtype=torch.bfloat16, device="cuda")
    qb = synth.queries(w_, 7, 300)
    q.qwm_update_query_stats(ctx, _bf(qb), 300, S, n, w, lam, ur)
    assert q.qwm_sync_status(ctx) == 0
    S64 = np.zeros((H, D, D)); n64 = np.zeros(H, np.int64)
    ow, olam, our, oU, _ = oracle.update_query_stats(qb, S64, n64, 16)
    gl = lam.cpu().numpy()
    assert np.all(np.abs(gl - olam) <= 1e-3 * np.abs(olam) + 1e-6 * np.abs(olam).max())
    gu = _f32(to_u16(ur))
    for h in range(H):
        M = S64[h] / n64[h]
        U = gu[h]
        assert np.abs(U.T @ U - np.eye(16)).max() < 1e-2
        for k in range(16):
            res = np.linalg.norm(M @ U[:, k] - olam[h, k] * U[:, k])
            assert res <= 5e-3 * olam[h, 0], (h, k, res)
        for k in range(8):
            assert U[:, k] @ oU[h][:, k] / np.linalg.norm(U[:, k]) > 0.999


@pytest.mark.parametrize("nq", [3, 1])
def test_basis_fewer_queries_than_rank(q, nq):
    """M of rank nq < r: the eigenvalue 0 has multiplicity 128 - nq.  No error is recorded, the
    nonzero eigenpairs match the oracle's, and the remaining columns are orthonormal vectors of the
    null space (any such basis is an eigenbasis there)."""
    w_ = synth.TINY
    H = w_.heads
    ctx = q.Context(heads=H, rank=8)
    S = torch.zeros(H, D, D, device="cuda"); n = torch.zeros(H, dtype=torch.int64, device="cuda")
    w = torch.empty(H, D, device="cuda"); lam = torch.empty(H, D, device="cuda")
    ur = torch.empty(H, D, 8, dtype=torch.bfloat16, device="cuda")
    qb = synth.queries(w_, 9, nq)
    q.qwm_update_query_stats(ctx, _bf(qb), nq, S, n, w, lam, ur)
    assert q.qwm_sync_status(ctx) == 0
    S64 = np.zeros((H, D, D)); n64 = np.zeros(H, np.int64)
    ow, olam, our, oU, _ = oracle.update_query_stats(qb, S64, n64, 8)
    gl = lam.cpu().numpy()
    assert np.all(np.abs(gl - olam) <= 1e-3 * np.abs(olam) + 1e-6 * np.abs(olam).max())
    gu = _f32(to_u16(ur))
    for h in range(H):
        U = gu[h]
        assert np.isfinite(U).all()
        assert np.abs(U.T @ U - np.eye(8)).max() < 1e-2
        for k in range(nq):
            assert U[:, k] @ oU[h][:, k] / np.linalg.norm(U[:, k]) > 0.999
        M = S64[h] / n64[h]
        for k in range(nq, 8):
            assert np.linalg.norm(M @ U[:, k]) <= 5e-3 * olam[h, 0], (h, k)


# ------------------------------------------------------------------ step 2a


@pytest.mark.parametrize("n,C,init", [(1024, 256, False), (1000, 64, False), (1024, 256, True)])
def test_kmeans_objective(q, n, C, init):
    w_ = synth.TINY
    H = w_.heads
    x = synth.keys(w_)[:, :n]
    ctx = q.Context(heads=H, n_centroids=C, top_m=min(4, C))
    init_np = None
    if init:
        init_np = np.stack([oracle.kmeans(x[h], C, None, 2)[0] for h in range(H)])
    cent = torch.empty(H, C, D, dtype=torch.bfloat16, device="cuda")
    q.qwm_fit_centroids(ctx, _bf(x), n, None if init_np is None else _bf(init_np), cent)
    assert q.qwm_sync_status(ctx) == 0
    for h in range(H):
        ref, _, _, _ = oracle.kmeans(x[h], C, None if init_np is None else init_np[h], 10)
        j_gpu = oracle.kmeans_objective(x[h], to_u16(cent[h]))
        j_ref = oracle.kmeans_objective(x[h], ref)
        assert abs(j_gpu - j_ref) <= 1e-3 * j_ref, (h, j_gpu, j_ref)


# ------------------------------------------------------------------ steps 2-4


# 1024-centroid cases: two heads of the ablation-shaped recipe (6 frames of 30 x 52 tokens), enough
# tokens for a 1024-centroid codebook; these run the kernels' streamed-codebook variants.
WIDE_W = synth.Workload("ablation-2-heads", 4, heads=2, frames=6, hs=30, ws=52, frames_per_chunk=3,
                        nq_stats=256, nq_attend=256, n_centroids=1024)


def test_kmeans_objective_past_the_kept_assignments(q):
    """A chunk longer than the 65,536 tokens per head whose assignments the context keeps between Lloyd
    iterations: every iteration then recomputes its cluster sums in full (152 CTAs on one head)."""
    n, C = 70000, 64
    x = np.ascontiguousarray(synth.keys(synth.P720, 0, 0, n)[:1])
    ctx = q.Context(heads=1, n_centroids=C, top_m=4)
    cent = torch.empty(1, C, D, dtype=torch.bfloat16, device="cuda")
    q.qwm_fit_centroids(ctx, _bf(x), n, None, cent)
    assert q.qwm_sync_status(ctx) == 0
    ref, _, _, _ = oracle.kmeans(x[0], C, None, 10)
    j_gpu = oracle.kmeans_objective(x[0], to_u16(cent[0]))
    j_ref = oracle.kmeans_objective(x[0], ref)
    assert abs(j_gpu - j_ref) <= 1e-3 * j_ref, (j_gpu, j_ref)


@pytest.mark.parametrize("C,warm", [(64, False), (256, True), (1024, False)], ids=["c64", "c256_warm", "c1024"])
def test_fit_centroids_kv_equals_two_fits(q, C, warm):
    """The paired call (the Value fit on the context's second stream with its own workspace) gives
    the two codebooks of two qwm_fit_centroids calls bit for bit, and the context stays usable for
    single fits afterwards."""
    H, n = 2, 2600
    k = _bf(synth.keys(WIDE_W)[:, :n]); v = _bf(synth.values(WIDE_W)[:, :n])
    ctx = q.Context(heads=H, n_centroids=C, top_m=4)
    init_k = init_v = None
    if warm:  # the previous chunk's codebooks as the starting points
        init_k = torch.empty(H, C, D, dtype=torch.bfloat16, device="cuda"); init_v = torch.empty_like(init_k)
        q.qwm_fit_centroids(ctx, _bf(synth.keys(WIDE_W)[:, n:2 * n]), n, None, init_k)
        q.qwm_fit_centroids(ctx, _bf(synth.values(WIDE_W)[:, n:2 * n]), n, None, init_v)
    ref_k = torch.empty(H, C, D, dtype=torch.bfloat16, device="cuda"); ref_v = torch.empty_like(ref_k)
    q.qwm_fit_centroids(ctx, k, n, init_k, ref_k)
    q.qwm_fit_centroids(ctx, v, n, init_v, ref_v)
    ck, cv = torch.empty_like(ref_k), torch.empty_like(ref_k)
    q.qwm_fit_centroids_kv(ctx, k, v, n, init_k, init_v, ck, cv)
    again = torch.empty_like(ref_k)
    q.qwm_fit_centroids(ctx, v, n, init_v, again)
    assert q.qwm_sync_status(ctx) == 0
    assert torch.equal(ck, ref_k) and torch.equal(cv, ref_v) and torch.equal(again, ref_v)
    with pytest.raises(q.QwmError) as e:   # one buffer for both codebooks
        q.qwm_fit_centroids_kv(ctx, k, v, n, init_k, init_v, ck, ck)
    assert e.value.status == q.QWM_ERR_ARG


def test_kmeans_objective_1024_centroids(q):
    H, n, C = 2, 2600, 1024
    x = synth.keys(WIDE_W)[:, :n]
    ctx = q.Context(heads=H, n_centroids=C, top_m=4)
    cent = torch.empty(H, C, D, dtype=torch.bfloat16, device="cuda")
    q.qwm_fit_centroids(ctx, _bf(x), n, None, cent)
    assert q.qwm_sync_status(ctx) == 0
    for h in range(H):
        ref, _, _, _ = oracle.kmeans(x[h], C, None, 10)
        j_gpu = oracle.kmeans_objective(x[h], to_u16(cent[h]))
        j_ref = oracle.kmeans_objective(x[h], ref)
        assert abs(j_gpu - j_ref) <= 1e-3 * j_ref, (h, j_gpu, j_ref)


def _upstream(q, w_, H, n, C=256, top_m=4, rank=8, psac=True, storage=0, gate=0):
    """GPU statistics and codebooks for a small case; returns numpy and device pieces."""
    k = synth.keys(w_)[:H, :n]; v = synth.values(w_)[:H, :n]
    ctx = q.Context(heads=H, n_centroids=C, top_m=top_m, rank=rank, storage=storage, psac_gate=gate)
    layer_S = torch.zeros(H, D, D, device="cuda"); n_ = torch.zeros(H, dtype=torch.int64, device="cuda")
    w = torch.empty(H, D, device="cuda"); lam = torch.empty(H, D, device="cuda")
    ur = torch.zeros(H, D, max(rank, 1), dtype=torch.bfloat16, device="cuda")
    if psac:
        qs = synth.queries(w_, -1, 256)[:H]
        q.qwm_update_query_stats(ctx, _bf(qs), 256, layer_S, n_, w, lam, ur if rank else None)
    ch = q.Chunk.empty(ctx, n)
    K, V = _bf(k), _bf(v)
    q.qwm_fit_centroids(ctx, K, n, None, ch.cent_k)
    q.qwm_fit_centroids(ctx, V, n, None, ch.cent_v)
    if psac and rank:
        ch.u_r.copy_(ur)
    return ctx, k, v, K, V, ch, (w if psac else None), (ch.u_r if psac and rank else None)


def _check_quantize(q, ctx, k, v, K, V, ch, w, ur, top_m, rank, M=None, Sn=None):
    H, n = k.shape[:2]
    dbg = dict(c_f32=torch.zeros(H, n, max(rank, 1), device="cuda"),
               cand=torch.zeros(H, n, top_m, dtype=torch.int32, device="cuda"),
               score=torch.zeros(H, n, device="cuda"))
    if M is None:
        q.qwm_quantize_kv(ctx, K, V, n, w, ur, ch, dbg)
    else:
        q.qwm_quantize_kv_full(ctx, K, V, n, Sn[0], Sn[1], ur, ch, dbg)
    assert q.qwm_sync_status(ctx) == 0
    assert ch.rank_eff == (rank if ur is not None else 0)
    stats = dict(k_ties=0, v_ties=0, k_edge=0, tokens=H * n)
    for h in range(H):
        wh = None if w is None else w[h].cpu().numpy().astype(np.float64)
        Mh = None if M is None else M[h].cpu().numpy().astype(np.float64)
        if Mh is not None:
            wh = np.diag(Mh).copy()
        urh = None if ur is None else to_u16(ur[h])[:, :rank]
        o = oracle.quantize_head(k[h], v[h], to_u16(ch.cent_k[h]), to_u16(ch.cent_v[h]), wh, urh,
                                 top_m=top_m, rank=rank if ur is not None else 0, M_full=Mh)
        gk = ch.k_idx[h].cpu().numpy().astype(np.int32)
        gv = ch.v_idx[h].cpu().numpy().astype(np.int32)
        s2 = o["score2"]; de = o["dq_edge"]; vd = o["vdist2"]
        k_tie = np.abs(s2[:, 1] - s2[:, 0]) <= TIE * np.abs(s2[:, 0])
        k_edge = np.abs(de[:, 1] - de[:, 0]) <= TIE * np.abs(de[:, 0])
        v_tie = np.abs(vd[:, 1] - vd[:, 0]) <= TIE * np.abs(vd[:, 0])
        bad_k = (gk != o["idx_k"]) & ~(k_tie | k_edge)
        bad_v = (gv != o["idx_v"]) & ~v_tie
        assert not bad_k.any(), f"head {h}: {bad_k.sum()} Key index mismatches outside ties"
        assert not bad_v.any(), f"head {h}: {bad_v.sum()} Value index mismatches outside ties"
        stats["k_ties"] += int(k_tie.sum()); stats["k_edge"] += int(k_edge.sum()); stats["v_ties"] += int(v_tie.sum())
        # candidate sets agree (as sets) wherever the boundary is not a tie
        gc = np.sort(dbg["cand"][h].cpu().numpy(), axis=1)
        oc = np.sort(o["cand"], axis=1)
        assert np.all((gc == oc).all(1) | k_edge)
        # re-encode with the GPU's indices: codes, scales and offsets bit-exact
        o2 = oracle.quantize_head(k[h], v[h], to_u16(ch.cent_k[h]), to_u16(ch.cent_v[h]), wh, urh,
                                  top_m=top_m, rank=rank if ur is not None else 0, force_idx_k=gk, force_idx_v=gv,
                                  M_full=Mh)
        for name in ("k_codes", "v_codes"):
            assert np.array_equal(getattr(ch, name)[h].cpu().numpy(), o2[name]), name
        for name in ("k_scale", "k_min", "v_scale", "v_min"):
            assert np.array_equal(to_u16(getattr(ch, name)[h]), o2[name]), name
        if ur is not None:
            cg = dbg["c_f32"][h].cpu().numpy()[:, :rank].astype(np.float64)
            cr = o2["c_real"]
            scale_ = np.maximum(np.abs(cr).max(1, keepdims=True), 1e-30)
            assert np.all(np.abs(cg - cr) <= 1e-3 * scale_)
            # INT8 encoding of the GPU's fp32 coefficients: bit-exact
            gc8 = ch.c[h].cpu().numpy()[:, :rank]
            gsc = to_u16(ch.c_scale[h])
            for i in range(n):
                c8, sc = oracle.int8_encode_token(cg[i].astype(np.float32))
                assert sc == gsc[i] and np.array_equal(c8, gc8[i]), i
    return stats


def test_quantize_tiny_with_psac(q):
    ctx, k, v, K, V, ch, w, ur = _upstream(q, synth.TINY, 2, 1024)
    st = _check_quantize(q, ctx, k, v, K, V, ch, w, ur, 4, 8)
    print("tie fractions", {key: val / st["tokens"] for key, val in st.items() if key != "tokens"})


def test_quantize_cold_start(q):
    ctx, k, v, K, V, ch, w, ur = _upstream(q, synth.TINY, 2, 1024, psac=False)
    _check_quantize(q, ctx, k, v, K, V, ch, None, None, 4, 8)


@pytest.mark.parametrize("n,C,top_m,rank", [(333, 64, 16, 16), (257, 128, 1, 0), (300, 256, 4, 8), (401, 256, 2, 8)])
def test_quantize_ragged_and_shapes(q, n, C, top_m, rank):
    ctx, k, v, K, V, ch, w, ur = _upstream(q, synth.TINY, 2, n, C=C, top_m=top_m, rank=rank)
    _check_quantize(q, ctx, k, v, K, V, ch, w, ur, top_m, rank)


@pytest.mark.parametrize("C,n,top_m", [(256, 1000, 4), (64, 700, 16), (1024, 2000, 4)])
def test_quantize_full_form_ranking(q, C, n, top_m):
    """English v2 §C.4 ablation: candidates ranked by (k - mu)^T M (k - mu) with the full Query second
    moment M (from the GPU statistics), the choice by the range score with w = diag(M)."""
    w_ = WIDE_W if C > 256 else synth.TINY
    H = 2
    k = synth.keys(w_)[:H, :n]; v = synth.values(w_)[:H, :n]
    ctx = q.Context(heads=H, n_centroids=C, top_m=top_m, rank=8)
    S = torch.zeros(H, D, D, device="cuda"); cnt = torch.zeros(H, dtype=torch.int64, device="cuda")
    w = torch.empty(H, D, device="cuda"); lam = torch.empty(H, D, device="cuda")
    ur = torch.zeros(H, D, 8, dtype=torch.bfloat16, device="cuda")
    q.qwm_update_query_stats(ctx, _bf(synth.queries(w_, -1, 256)[:H]), 256, S, cnt, w, lam, ur)
    # the library forms M = S / n in fp32 (IEEE division); the oracle ranks with the same values
    M = torch.from_numpy(S.cpu().numpy() / cnt.cpu().numpy().astype(np.float32)[:, None, None])
    ch = q.Chunk.empty(ctx, n)
    K, V = _bf(k), _bf(v)
    q.qwm_fit_centroids(ctx, K, n, None, ch.cent_k)
    q.qwm_fit_centroids(ctx, V, n, None, ch.cent_v)
    ch.u_r.copy_(ur)
    st = _check_quantize(q, ctx, k, v, K, V, ch, None, ch.u_r, top_m, 8, M=M, Sn=(S, cnt))
    print("tie fractions", {key: val / st["tokens"] for key, val in st.items() if key != "tokens"})


@pytest.mark.parametrize("n,top_m,rank", [(2600, 4, 8), (1500, 16, 16), (1100, 1, 0)])
def test_quantize_1024_centroids(q, n, top_m, rank):
    ctx, k, v, K, V, ch, w, ur = _upstream(q, WIDE_W, 2, n, C=1024, top_m=top_m, rank=rank)
    assert ch.k_idx.element_size() == 2
    st = _check_quantize(q, ctx, k, v, K, V, ch, w, ur, top_m, rank)
    print("tie fractions", {key: val / st["tokens"] for key, val in st.items() if key != "tokens"})


@pytest.mark.parametrize("C", [256, 1024])
def test_quantize_duplicated_codebook(q, C):
    """Every centroid repeated 8 times: each token's candidate window holds at least 8 exactly tied
    centroids, so the exact fallback resolves every token (for 1024 centroids the window reaches past
    the kernel's list and the whole codebook is searched).  Ties go to the lower index on both sides."""
    H, n, M = 2, (1100 if C > 256 else 1000), 4
    w_ = WIDE_W if C > 256 else synth.TINY
    ctx, k, v, K, V, ch, w, ur = _upstream(q, w_, H, n, C=C, top_m=M, rank=8)
    for cb in (ch.cent_k, ch.cent_v):
        cb.copy_(cb[:, ::8].repeat_interleave(8, dim=1))
    q.qwm_quantize_kv(ctx, K, V, n, w, ur, ch)
    assert q.qwm_sync_status(ctx) == 0
    for h in range(H):
        wh = w[h].cpu().numpy().astype(np.float64)
        o = oracle.quantize_head(k[h], v[h], to_u16(ch.cent_k[h]), to_u16(ch.cent_v[h]), wh,
                                 to_u16(ur[h])[:, :8], top_m=M, rank=8)
        gk = ch.k_idx[h].cpu().numpy().astype(np.int32)
        gv = ch.v_idx[h].cpu().numpy().astype(np.int32)
        # near-ties between distinct rows (not the planted exact copies) may go either way
        uk, uv = _f32(to_u16(ch.cent_k[h][::8])), _f32(to_u16(ch.cent_v[h][::8]))
        kx, vx = _f32(k[h]), _f32(v[h])
        dk = np.sort(((kx[:, None, :] - uk[None]) ** 2 * wh).sum(-1), axis=1)
        dv = np.sort(((vx[:, None, :] - uv[None]) ** 2).sum(-1), axis=1)
        s2 = o["score2"]
        k_free = (np.abs(dk[:, 1] - dk[:, 0]) <= TIE * dk[:, 0]) | (np.abs(s2[:, 1] - s2[:, 0]) <= TIE * np.abs(s2[:, 0]))
        v_free = np.abs(dv[:, 1] - dv[:, 0]) <= TIE * dv[:, 0]
        assert np.all((gk == o["idx_k"]) | k_free), (h, int(((gk != o["idx_k"]) & ~k_free).sum()))
        assert np.all((gv == o["idx_v"]) | v_free), (h, int(((gv != o["idx_v"]) & ~v_free).sum()))
        assert np.all(gk % 8 < M) and np.all(gv % 8 == 0)  # the lowest copies win


@pytest.mark.parametrize("gate,n", [(0, 1000), (1, 1000), (1, 300)])
def test_quantize_compact_storage_and_psac_gate(q, gate, n):
    """The paper's compact metadata (8-bit step, 2-bit zero-point, power-of-two second-level scale per
    128-token tile) bit-exact given the indices; with the gate, C dropped exactly where it does not lower
    the w-weighted error (decisions within a relative 1e-3 of a tie may go either way)."""
    H, M, R = 2, 4, 8
    ctx, k, v, K, V, ch, w, ur = _upstream(q, synth.TINY, H, n, storage=1, gate=gate)
    assert ch.compact
    dbg = dict(c_f32=torch.zeros(H, n, R, device="cuda"), cand=torch.zeros(H, n, M, dtype=torch.int32, device="cuda"),
               score=torch.zeros(H, n, device="cuda"), gate_err=torch.zeros(H, n, 2, device="cuda"))
    q.qwm_quantize_kv(ctx, K, V, n, w, ur, ch, dbg)
    assert q.qwm_sync_status(ctx) == 0
    for h in range(H):
        wh = w[h].cpu().numpy().astype(np.float64)
        urh = to_u16(ur[h])[:, :R]
        gk = ch.k_idx[h].cpu().numpy().astype(np.int32); gv = ch.v_idx[h].cpu().numpy().astype(np.int32)
        o = oracle.quantize_head(k[h], v[h], to_u16(ch.cent_k[h]), to_u16(ch.cent_v[h]), wh, urh, top_m=M, rank=R,
                                 storage=1, psac_gate=gate, force_idx_k=gk, force_idx_v=gv)
        for name in ("k_codes", "v_codes", "k_s8", "v_s8"):
            assert np.array_equal(getattr(ch, name)[h].cpu().numpy(), o[name]), name
        for name in ("k_zp", "v_zp"):
            assert np.array_equal(getattr(ch, name)[h].cpu().numpy()[:n], o[name]), name
        for name in ("k_sigma", "v_sigma"):
            assert np.array_equal(to_u16(getattr(ch, name)[h]), o[name]), name
        cg = dbg["c_f32"][h].cpu().numpy().astype(np.float64)
        cr = o["c_real"]
        assert np.all(np.abs(cg - cr) <= 1e-3 * np.maximum(np.abs(cr).max(1, keepdims=True), 1e-30))
        gc8, gsc = ch.c[h].cpu().numpy()[:, :R], to_u16(ch.c_scale[h])
        e0, e1 = o["gate_err"][:, 0], o["gate_err"][:, 1]
        near = np.abs(e1 - e0) <= 1e-3 * np.maximum(e0, 1e-30)
        for i in range(n):
            c8, sc = oracle.int8_encode_token(cg[i].astype(np.float32))
            kept = gsc[i] == sc and np.array_equal(gc8[i], c8)
            dropped = gsc[i] == 0 and not gc8[i].any()
            assert kept or (gate and dropped), i
            if gate and not near[i] and sc != 0:
                assert kept == bool(e1[i] < e0[i]), (i, e0[i], e1[i])


@pytest.mark.parametrize("C", [256, 1024])
def test_attend_and_decode_compact_chunk(q, C):
    H, n = 2, (1000 if C == 256 else 2600)
    ctx, k, v, K, V, ch, w, ur = _upstream(q, WIDE_W if C > 256 else synth.TINY, H, n, C=C, storage=1, gate=1)
    q.qwm_quantize_kv(ctx, K, V, n, w, ur, ch)
    nq = 300
    qa = synth.queries(synth.TINY, 5, nq)
    out = torch.empty(H, nq, D, dtype=torch.float32, device="cuda")
    q.qwm_attend(ctx, _bf(qa), nq, [ch], 1 / math.sqrt(D), out)
    kh = torch.empty(H, n, D, dtype=torch.bfloat16, device="cuda"); vh = torch.empty_like(kh)
    q.qwm_dequantize(ctx, ch, kh, vh)
    assert q.qwm_sync_status(ctx) == 0
    for h in range(H):
        c = chunk_head(ch, h)
        ref = oracle.attend_rows(qa[h], np.arange(nq), [c], 1 / math.sqrt(D))
        assert _attn_err(out[h].cpu().numpy().astype(np.float64), ref) <= 2e-2
        _, _, k64, v64 = oracle.dequantize_head(c)
        for got, ref64, key in ((kh[h], k64, True), (vh[h], v64, False)):
            g = (to_u16(got).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
            slack = 2.0 ** -20 * decode_term_magnitude(c, key)
            assert (bf16_ulp_close(to_u16(got), ref64) | (np.abs(g - ref64) <= slack)).all()


# ------------------------------------------------------------------ step 5', step 5


def _packed(q, n=1024, H=2, psac=True, C=256, rank=8):
    ctx, k, v, K, V, ch, w, ur = _upstream(q, WIDE_W if C > 256 else synth.TINY, H, n, C=C, rank=rank, psac=psac)
    q.qwm_quantize_kv(ctx, K, V, n, w, ur, ch)
    assert q.qwm_sync_status(ctx) == 0
    return ctx, ch


@pytest.mark.parametrize("psac,C,n", [(True, 256, 1024), (False, 256, 1024), (True, 1024, 2000)])
def test_dequantize_within_one_bf16_step(q, psac, C, n):
    ctx, ch = _packed(q, n=n, psac=psac, C=C)
    H, n = 2, ch.n_tokens
    kh = torch.empty(H, n, D, dtype=torch.bfloat16, device="cuda"); vh = torch.empty_like(kh)
    q.qwm_dequantize(ctx, ch, kh, vh)
    assert q.qwm_sync_status(ctx) == 0
    for h in range(H):
        c = chunk_head(ch, h)
        _, _, k64, v64 = oracle.dequantize_head(c)
        # one bf16 step, plus the fp32 evaluation error where the decoder's sum cancels
        for got, ref, key in ((kh[h], k64, True), (vh[h], v64, False)):
            g = (to_u16(got).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
            slack = 2.0 ** -20 * decode_term_magnitude(c, key)
            assert (bf16_ulp_close(to_u16(got), ref) | (np.abs(g - ref) <= slack)).all()


def test_dequantize_chunks_one_launch(q):
    """Several chunks (cold start without PSAC, then PSAC chunks with their own bases, ragged sizes)
    decoded in one launch into [H][sum N][d]: identical to decoding each chunk alone, and each
    chunk's rows within one bf16 step of the oracle's decoder (plus the cancellation slack)."""
    w_ = synth.TINY
    H = 2
    ctx = q.Context(heads=H)
    from bit_kv_cache_qsac_gb300 import stream
    layer = stream.CompressedLayer(ctx)
    kk, vv = synth.keys(w_), synth.values(w_)
    parts = [(0, 300), (300, 700), (700, 1024)]
    for i, (a, b) in enumerate(parts):
        if i > 0:
            layer.fold_queries(_bf(synth.queries(w_, 30 + i, 128)))
        layer.append_chunk(_bf(np.ascontiguousarray(kk[:, a:b])), _bf(np.ascontiguousarray(vv[:, a:b])))
    total = sum(c.n_tokens for c in layer.chunks)
    kh = torch.empty(H, total, D, dtype=torch.bfloat16, device="cuda"); vh = torch.empty_like(kh)
    q.qwm_dequantize_chunks(ctx, layer.chunks, kh, vh)
    assert q.qwm_sync_status(ctx) == 0
    row = 0
    for i, ch in enumerate(layer.chunks):
        k1, v1 = layer.dequantize(i)
        n = ch.n_tokens
        assert torch.equal(kh[:, row:row + n], k1) and torch.equal(vh[:, row:row + n], v1)
        for h in range(H):
            c = chunk_head(ch, h)
            _, _, k64, v64 = oracle.dequantize_head(c)
            for got, ref, key in ((kh[h, row:row + n], k64, True), (vh[h, row:row + n], v64, False)):
                g = (to_u16(got).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
                slack = 2.0 ** -20 * decode_term_magnitude(c, key)
                assert (bf16_ulp_close(to_u16(got), ref) | (np.abs(g - ref) <= slack)).all()
        row += n


def _attn_err(got, ref):
    return np.abs(got - ref).max() / math.sqrt(np.mean(ref ** 2))


@pytest.mark.parametrize("nq", [256, 200, 1])
def test_attend_tiny(q, nq):
    ctx, ch = _packed(q)
    H = 2
    qa = synth.queries(synth.TINY, 0, nq)
    out = torch.empty(H, nq, D, dtype=torch.float32, device="cuda")
    q.qwm_attend(ctx, _bf(qa), nq, [ch], 1 / math.sqrt(D), out)
    assert q.qwm_sync_status(ctx) == 0
    for h in range(H):
        ref = oracle.attend_rows(qa[h], np.arange(nq), [chunk_head(ch, h)], 1 / math.sqrt(D))
        err = _attn_err(out[h].cpu().numpy().astype(np.float64), ref)
        assert err <= 2e-2, err


@pytest.mark.parametrize("rank,C,n", [(16, 256, 1024), (12, 128, 777), (5, 64, 300), (0, 256, 513),
                                       (8, 1024, 2600), (16, 1024, 1500)])
def test_attend_psac_ranks(q, rank, C, n):
    """PSAC ranks above 8 take the kernel's 32-column second-MMA operands (ranks 12 and 16, with
    the coefficient rows read byte by byte for 12); ranks up to 8 the 16-column ones."""
    ctx, ch = _packed(q, n=n, C=C, rank=rank)
    H, nq = 2, 300
    qa = synth.queries(synth.TINY, 1, nq)
    out = torch.empty(H, nq, D, dtype=torch.float32, device="cuda")
    q.qwm_attend(ctx, _bf(qa), nq, [ch], 1 / math.sqrt(D), out)
    assert q.qwm_sync_status(ctx) == 0
    for h in range(H):
        ref = oracle.attend_rows(qa[h], np.arange(nq), [chunk_head(ch, h)], 1 / math.sqrt(D))
        assert _attn_err(out[h].cpu().numpy().astype(np.float64), ref) <= 2e-2


@pytest.mark.parametrize("rank,C,n", [(5, 64, 300), (7, 256, 513), (11, 128, 777), (12, 128, 777),
                                       (16, 256, 1024)])
def test_dequantize_psac_ranks(q, rank, C, n):
    """The Key decoder's PSAC term on warp-level MMAs at odd and even ranks on both sides of 8: ranks up
    to 8 take the K = 8 products, above 8 the K = 16 ones; an odd rank reads the basis in 16-bit
    halves.  Every element within one bf16 step of the oracle's decoder (plus the cancellation slack)."""
    ctx, ch = _packed(q, n=n, C=C, rank=rank)
    H = 2
    kh = torch.empty(H, n, D, dtype=torch.bfloat16, device="cuda"); vh = torch.empty_like(kh)
    q.qwm_dequantize(ctx, ch, kh, vh)
    assert q.qwm_sync_status(ctx) == 0
    for h in range(H):
        c = chunk_head(ch, h)
        _, _, k64, v64 = oracle.dequantize_head(c)
        for got, ref, key in ((kh[h], k64, True), (vh[h], v64, False)):
            g = (to_u16(got).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
            slack = 2.0 ** -20 * decode_term_magnitude(c, key)
            assert (bf16_ulp_close(to_u16(got), ref) | (np.abs(g - ref) <= slack)).all()


def test_attend_growing_logits(q):
    """A hand-built chunk whose logits rise steadily along the keys (about 10 log2 units per tile),
    so the softmax raises its running maximum many times, inside tiles and across them (rescaling
    its sum, O and the P chunks already written).  Every decoded key is an integer vector and every
    Query a multiple of 1/8, so the logits are exact in the kernel's fp16 operands and the only
    differences from the oracle are the rounding of P and of the exponentials."""
    H, n, C, nq = 2, 1024, 256, 256
    ctx = q.Context(heads=H, n_centroids=C, rank=0)
    ch = q.Chunk.empty(ctx, n)
    rng = np.random.default_rng(7)
    u = np.where(rng.random(D) < 0.5, -1.0, 1.0)
    ck = np.stack([np.round(20.0 * np.arange(C) / C)[:, None] * u[None, :]] * H)    # centroid j ~ (20 j / C) u
    cv = rng.integers(-3, 4, size=(H, C, D)).astype(np.float64)
    idx = np.broadcast_to(np.arange(n) // (n // C), (H, n)).astype(np.uint8)
    for name in ("k_codes", "v_codes"):
        getattr(ch, name).zero_()
    for name in ("k_scale", "k_min", "v_scale", "v_min"):
        getattr(ch, name).zero_()
    ch.k_idx.copy_(torch.from_numpy(idx.copy())); ch.v_idx.copy_(torch.from_numpy(idx.copy()))
    ch.cent_k.copy_(torch.from_numpy(ck).to(torch.bfloat16)); ch.cent_v.copy_(torch.from_numpy(cv).to(torch.bfloat16))
    # the stored codebooks the attention reads (integers: exact in fp16)
    ch.cent_k16.copy_(torch.from_numpy(ck).to(torch.float16)); ch.cent_v16.copy_(torch.from_numpy(cv).to(torch.float16))
    qf = 0.25 * u[None, None, :] + 0.125 * rng.integers(-2, 3, size=(H, nq, D))
    qa = to_u16(torch.from_numpy(qf).to(torch.bfloat16))
    out = torch.empty(H, nq, D, dtype=torch.float32, device="cuda")
    q.qwm_attend(ctx, _bf(qa), nq, [ch], 1 / math.sqrt(D), out)
    assert q.qwm_sync_status(ctx) == 0
    for h in range(H):
        ref = oracle.attend_rows(qa[h], np.arange(nq), [chunk_head(ch, h)], 1 / math.sqrt(D))
        assert _attn_err(out[h].cpu().numpy().astype(np.float64), ref) <= 2e-3


@pytest.mark.parametrize("n,nq", [(1000, 300), (128, 1), (77, 64)])
def test_attend_bf16_chunk_alone(q, n, nq):
    """The chunk still being generated, alone: its bf16 rows attend as they are."""
    H = 2
    k = synth.keys(WIDE_W)[:H, :n]; v = synth.values(WIDE_W)[:H, :n]
    ctx = q.Context(heads=H)
    act = q.ActiveChunk(_bf(k), _bf(v))
    qa = synth.queries(WIDE_W, 3, nq)
    out = torch.empty(H, nq, D, dtype=torch.float32, device="cuda")
    q.qwm_attend(ctx, _bf(qa), nq, [act], 1 / math.sqrt(D), out)
    assert q.qwm_sync_status(ctx) == 0
    for h in range(H):
        ref = oracle.attend_rows(qa[h], np.arange(nq), [dict(k_raw=k[h], v_raw=v[h])], 1 / math.sqrt(D))
        assert _attn_err(out[h].cpu().numpy().astype(np.float64), ref) <= 2e-2


@pytest.mark.parametrize("tpf", [0, 256, 100])
def test_attend_packed_history_and_causal_active_chunk(q, tpf):
    """Packed history (1,024 tokens, PSAC) plus the chunk being generated (600 bf16 tokens) in one
    softmax; with tpf > 0 Query row i (token i of the active chunk) sees only the active chunk's frames
    up to its own."""
    ctx, ch = _packed(q)
    H, na = 2, 600
    k = synth.keys(WIDE_W)[:H, 2000:2000 + na]; v = synth.values(WIDE_W)[:H, 2000:2000 + na]
    act = q.ActiveChunk(_bf(np.ascontiguousarray(k)), _bf(np.ascontiguousarray(v)), causal_tpf=tpf)
    qa = synth.queries(WIDE_W, 4, na)
    out = torch.empty(H, na, D, dtype=torch.float32, device="cuda")
    q.qwm_attend(ctx, _bf(qa), na, [ch, act], 1 / math.sqrt(D), out)
    assert q.qwm_sync_status(ctx) == 0
    for h in range(H):
        ref = oracle.attend_rows(qa[h], np.arange(na),
                                 [chunk_head(ch, h), dict(k_raw=k[h], v_raw=v[h], causal_tpf=tpf)], 1 / math.sqrt(D))
        assert _attn_err(out[h].cpu().numpy().astype(np.float64), ref) <= 2e-2


@pytest.mark.parametrize("scale", [1e-6, 1e-3])
def test_attend_softmax_scale_and_padded_rows(q, scale):
    """A ragged chunk (513 tokens: 4 full tiles and one of a single row) at softmax scales far below
    1/sqrt(d): the 127 rows that pad the last tile get weight exactly 0 whatever the scale (at 1e-6
    the softmax is almost flat, so weight left on the zero pad rows would shrink O by ~20%)."""
    ctx, ch = _packed(q, n=513)
    H, nq = 2, 130
    qa = synth.queries(synth.TINY, 2, nq)
    out = torch.empty(H, nq, D, dtype=torch.float32, device="cuda")
    q.qwm_attend(ctx, _bf(qa), nq, [ch], scale, out)
    assert q.qwm_sync_status(ctx) == 0
    for h in range(H):
        ref = oracle.attend_rows(qa[h], np.arange(nq), [chunk_head(ch, h)], scale)
        assert _attn_err(out[h].cpu().numpy().astype(np.float64), ref) <= 2e-2


def test_attend_fp16_range_errors(q):
    """A Query element or an element of the chunk being generated beyond the fp16 range (the
    tensor cores' operand type) records QWM_ERR_RANGE; elements inside it do not."""
    ctx, ch = _packed(q)
    H, nq = 2, 64
    qa = synth.queries(synth.TINY, 3, nq)
    out = torch.empty(H, nq, D, dtype=torch.float32, device="cuda")
    big = synth.f32_to_bf16_bits(np.array([1.0e5], np.float32))[0]
    edge = synth.f32_to_bf16_bits(np.array([65280.0], np.float32))[0]   # the largest bf16 below 65504
    qb = qa.copy(); qb[1, 7, 33] = big
    q.qwm_attend(ctx, _bf(qb), nq, [ch], 1 / math.sqrt(D), out)
    assert q.qwm_sync_status(ctx) == q.QWM_ERR_RANGE
    qb = qa.copy(); qb[1, 7, 33] = edge
    q.qwm_attend(ctx, _bf(qb), nq, [ch], 1 / math.sqrt(D), out)
    assert q.qwm_sync_status(ctx) == 0
    k = synth.keys(WIDE_W)[:H, :200].copy(); v = synth.values(WIDE_W)[:H, :200].copy()
    v[0, 150, 3] = big
    act = q.ActiveChunk(_bf(k), _bf(v))
    q.qwm_attend(ctx, _bf(qa), nq, [ch, act], 1 / math.sqrt(D), out)
    assert q.qwm_sync_status(ctx) == q.QWM_ERR_RANGE


def test_attend_expired_wait_recovers(q):
    """The test hook makes one bounded wait of the attention kernel run out: the call reports
    QWM_ERR_DEVICE_TIMEOUT, and the GPU and the library stay usable (a normal call that follows
    gives the oracle's output)."""
    ctx, ch = _packed(q)
    H, nq = 2, 256
    qa = synth.queries(synth.TINY, 5, nq)
    out = torch.empty(H, nq, D, dtype=torch.float32, device="cuda")
    hook = q.Context(heads=H, test_flags=q.QWM_TEST_EXPIRE_WAIT)
    q.qwm_attend(hook, _bf(qa), nq, [ch], 1 / math.sqrt(D), out)
    assert q.qwm_sync_status(hook) == q.QWM_ERR_DEVICE_TIMEOUT
    assert q.qwm_sync_status(hook) == 0          # the status word was cleared
    q.qwm_attend(ctx, _bf(qa), nq, [ch], 1 / math.sqrt(D), out)
    assert q.qwm_sync_status(ctx) == 0
    for h in range(H):
        ref = oracle.attend_rows(qa[h], np.arange(nq), [chunk_head(ch, h)], 1 / math.sqrt(D))
        assert _attn_err(out[h].cpu().numpy().astype(np.float64), ref) <= 2e-2


def test_attend_several_chunks_mixed_rank(q):
    """A cold-start chunk (no PSAC) followed by PSAC chunks with different bases and a ragged size."""
    w_ = synth.TINY
    H = 2
    ctx = q.Context(heads=H)
    from bit_kv_cache_qsac_gb300 import stream
    layer = stream.CompressedLayer(ctx)
    kk, vv = synth.keys(w_), synth.values(w_)
    parts = [(0, 300), (300, 700), (700, 1024)]
    for i, (a, b) in enumerate(parts):
        if i > 0:
            layer.fold_queries(_bf(synth.queries(w_, 10 + i, 128)))
        layer.append_chunk(_bf(np.ascontiguousarray(kk[:, a:b])), _bf(np.ascontiguousarray(vv[:, a:b])))
    assert [c.rank_eff for c in layer.chunks] == [0, 8, 8]
    qa = synth.queries(w_, 0, 96)
    out = layer.attend(_bf(qa))
    assert layer.check() == 0
    for h in range(H):
        ref = oracle.attend_rows(qa[h], np.arange(96), [chunk_head(c, h) for c in layer.chunks], 1 / math.sqrt(D))
        assert _attn_err(out[h].cpu().numpy().astype(np.float64), ref) <= 2e-2


def test_stream_step_matches_step(q):
    """The pipelined schedule (fold each step's Queries beside its attention) does the same work as
    folding the previous step's Queries before the packing: identical chunks and outputs."""
    w_ = synth.TINY
    H = w_.heads
    from bit_kv_cache_qsac_gb300 import stream
    kk, vv = synth.keys(w_), synth.values(w_)
    parts = [(0, 300), (300, 700), (700, 1024)]
    qs = [_bf(synth.queries(w_, 20 + i, 96)) for i in range(len(parts))]
    ka = q.Context(heads=H)
    kb = q.Context(heads=H)
    la, lb = stream.CompressedLayer(ka), stream.CompressedLayer(kb)
    outs_a, outs_b = [], []
    for i, (a, b) in enumerate(parts):
        k_ = _bf(np.ascontiguousarray(kk[:, a:b]))
        v_ = _bf(np.ascontiguousarray(vv[:, a:b]))
        outs_a.append(la.step(qs[i - 1] if i > 0 else None, k_, v_, qs[i]).clone())
        outs_b.append(lb.stream_step(k_, v_, qs[i]).clone())
    torch.cuda.synchronize()
    assert la.check() == 0 and lb.check() == 0
    assert [c.rank_eff for c in lb.chunks] == [0, 8, 8]
    for oa, ob in zip(outs_a, outs_b):
        assert torch.equal(oa, ob)
    for ca, cb in zip(la.chunks, lb.chunks):
        for name in ("k_idx", "v_idx", "k_codes", "v_codes", "c", "c_scale", "u_r"):
            assert torch.equal(getattr(ca, name), getattr(cb, name)), name
    # lb has also folded the last step's Queries: one more batch than la
    assert int(lb.n[0]) == int(la.n[0]) + 96


@pytest.mark.parametrize("with_active", [False, True], ids=["packed", "packed_then_active"])
def test_attend_merge_parts(q, with_active):
    """Two calls of qwm_attend_merge -- the first two packed chunks, then the third (and the chunk being
    generated, block-causal) merged in -- against the oracle over the union: the output within the
    attention's bar, each call's log-sum-exp within 0.02 (log2 units) of the oracle's; and against
    one call over the union: the same output and log-sum-exp up to the merge's fp32 rounding."""
    w_ = synth.TINY
    H = 2
    ctx = q.Context(heads=H)
    from bit_kv_cache_qsac_gb300 import stream
    layer = stream.CompressedLayer(ctx)
    kk, vv = synth.keys(w_), synth.values(w_)
    for i, (a, b) in enumerate([(0, 300), (300, 700), (700, 1024)]):
        if i > 0:
            layer.fold_queries(_bf(synth.queries(w_, 40 + i, 128)))
        layer.append_chunk(_bf(np.ascontiguousarray(kk[:, a:b])), _bf(np.ascontiguousarray(vv[:, a:b])))
    nq, tpf = 300, 100
    qa = synth.queries(WIDE_W, 5, nq)
    part_b = [layer.chunks[2]]
    ka = kv = None
    if with_active:
        ka = synth.keys(WIDE_W)[:H, 3000:3000 + nq]; kv = synth.values(WIDE_W)[:H, 3000:3000 + nq]
        part_b.append(q.ActiveChunk(_bf(np.ascontiguousarray(ka)), _bf(np.ascontiguousarray(kv)), causal_tpf=tpf))
    scale = 1 / math.sqrt(D)
    out = torch.empty(H, nq, D, dtype=torch.float32, device="cuda"); lse = torch.empty(H, nq, device="cuda")
    q.qwm_attend_merge(ctx, _bf(qa), nq, layer.chunks[:2], scale, out, lse, False)
    lse_a = lse.clone()
    q.qwm_attend_merge(ctx, _bf(qa), nq, part_b, scale, out, lse, True)
    one = torch.empty_like(out); lse1 = torch.empty_like(lse)
    q.qwm_attend_merge(ctx, _bf(qa), nq, layer.chunks[:2] + part_b, scale, one, lse1, False)
    assert q.qwm_sync_status(ctx) == 0
    for h in range(H):
        heads = [chunk_head(c, h) for c in layer.chunks]
        union = heads + ([dict(k_raw=ka[h], v_raw=kv[h], causal_tpf=tpf)] if with_active else [])
        ref, ref_lse = oracle.attend_rows(qa[h], np.arange(nq), union, scale, with_lse=True)
        _, ref_lse_a = oracle.attend_rows(qa[h], np.arange(nq), heads[:2], scale, with_lse=True)
        assert _attn_err(out[h].cpu().numpy().astype(np.float64), ref) <= 2e-2
        assert np.abs(lse[h].cpu().numpy() - ref_lse).max() <= 0.02
        assert np.abs(lse_a[h].cpu().numpy() - ref_lse_a).max() <= 0.02
    # each call rounds its weights P to fp16 relative to its own running maximum, so the two results'
    # weights differ by up to 2^-11 relative: O by at most about 2 * 2^-11 of its largest entries
    assert (out - one).abs().max().item() <= 1e-3 * one.abs().max().item()
    assert (lse - lse1).abs().max().item() <= 1e-5 * lse1.abs().max().item() + 1e-5


def test_stream_step_overlap_matches(q):
    """The overlapped schedule (history attention beside the new chunk's fits and packing, then the
    new chunk merged in) packs identical chunks and gives the sequential schedule's outputs up to
    the merge's rounding."""
    w_ = synth.TINY
    H = w_.heads
    from bit_kv_cache_qsac_gb300 import stream
    kk, vv = synth.keys(w_), synth.values(w_)
    parts = [(0, 300), (300, 700), (700, 1024)]
    qs = [_bf(synth.queries(w_, 20 + i, 96)) for i in range(len(parts))]
    la, lb = stream.CompressedLayer(q.Context(heads=H)), stream.CompressedLayer(q.Context(heads=H))
    outs_a, outs_b = [], []
    for i, (a, b) in enumerate(parts):
        k_ = _bf(np.ascontiguousarray(kk[:, a:b]))
        v_ = _bf(np.ascontiguousarray(vv[:, a:b]))
        outs_a.append(la.stream_step(k_, v_, qs[i]).clone())
        outs_b.append(lb.stream_step(k_, v_, qs[i], overlap=True).clone())
    torch.cuda.synchronize()
    assert la.check() == 0 and lb.check() == 0
    assert torch.equal(outs_a[0], outs_b[0])   # no history: the same single call
    for oa, ob in zip(outs_a[1:], outs_b[1:]):   # the fp16 weights' rounding, as in test_attend_merge_parts
        assert (oa - ob).abs().max().item() <= 1e-3 * oa.abs().max().item()
    for ca, cb in zip(la.chunks, lb.chunks):
        for name in ("k_idx", "v_idx", "k_codes", "v_codes", "c", "c_scale", "u_r"):
            assert torch.equal(getattr(ca, name), getattr(cb, name)), name


def test_bad_arguments_raise(q):
    ctx = q.Context(heads=2)
    x = torch.zeros(2, 300, D, dtype=torch.bfloat16, device="cuda")
    cent = torch.empty(2, 256, D, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(q.QwmError) as e:
        q.qwm_fit_centroids(ctx, x[:, :200].contiguous(), 200, None, cent)   # fewer tokens than centroids
    assert e.value.status == q.QWM_ERR_SHAPE
    lib = q.raw_library()
    bad = x.data_ptr() + 2   # misaligned
    assert lib.qwm_fit_centroids(ctx.handle, bad, 300, None, cent.data_ptr(), None) == q.QWM_ERR_ALIGN
    with pytest.raises(ValueError):
        q.qwm_fit_centroids(ctx, x, 299, None, cent)
    assert q.qwm_sync_status(ctx) == 0


# ------------------------------------------------------------------ edge cases


def test_edge_empty_inputs_and_limits(q):
    """Empty chunks and Query sets, a single-token chunk, one head, the 128-chunk limit of one call."""
    H = 1
    ctx = q.Context(heads=H, n_centroids=64, top_m=4, rank=8)
    k = synth.keys(synth.TINY)[:H, :256]; v = synth.values(synth.TINY)[:H, :256]
    K, V = _bf(k), _bf(v)
    # a codebook from 256 tokens, then chunks of 0, 1 and 17 tokens packed with it
    full = q.Chunk.empty(ctx, 256)
    q.qwm_fit_centroids(ctx, K, 256, None, full.cent_k)
    q.qwm_fit_centroids(ctx, V, 256, None, full.cent_v)
    chunks = []
    for n in (0, 1, 17):
        ch = q.Chunk.empty(ctx, n)
        ch.cent_k.copy_(full.cent_k); ch.cent_v.copy_(full.cent_v)
        q.qwm_quantize_kv(ctx, K[:, :n].contiguous(), V[:, :n].contiguous(), n, None, None, ch)
        chunks.append(ch)
    assert q.qwm_sync_status(ctx) == 0
    qa = synth.queries(synth.TINY, 6, 40)[:H]
    out = torch.empty(H, 40, D, dtype=torch.float32, device="cuda")
    q.qwm_attend(ctx, _bf(qa), 40, chunks, 1 / math.sqrt(D), out)       # the empty chunk is skipped
    assert q.qwm_sync_status(ctx) == 0
    ref = oracle.attend_rows(qa[0], np.arange(40), [chunk_head(c, 0) for c in chunks[1:]], 1 / math.sqrt(D))
    assert _attn_err(out[0].cpu().numpy().astype(np.float64), ref) <= 2e-2
    q.qwm_attend(ctx, _bf(qa[:, :0].copy()), 0, chunks, 1 / math.sqrt(D), out[:, :0])   # no Queries: a no-op
    with pytest.raises(q.QwmError) as e:
        q.qwm_attend(ctx, _bf(qa), 40, chunks[:1], 1 / math.sqrt(D), out)   # no key at all
    assert e.value.status == q.QWM_ERR_SHAPE
    kh = torch.empty(H, 0, D, dtype=torch.bfloat16, device="cuda")
    q.qwm_dequantize(ctx, chunks[0], kh, kh.clone())
    # 128 chunks of 2 tokens each (the most one call takes), then 129 (rejected)
    many = [chunks[2]] * 64 + [chunks[1]] * 64
    q.qwm_attend(ctx, _bf(qa), 40, many, 1 / math.sqrt(D), out)
    assert q.qwm_sync_status(ctx) == 0
    ref = oracle.attend_rows(qa[0], np.arange(40), [chunk_head(c, 0) for c in many], 1 / math.sqrt(D))
    assert _attn_err(out[0].cpu().numpy().astype(np.float64), ref) <= 2e-2
    with pytest.raises(q.QwmError):
        q.qwm_attend(ctx, _bf(qa), 40, many + [chunks[1]], 1 / math.sqrt(D), out)
