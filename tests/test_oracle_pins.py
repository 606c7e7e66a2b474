"""Pins of the CPU oracle to facts that do not come from the oracle itself.

Each test ties one oracle function to a closed form, a special case, a
library routine (numpy.linalg.eigh, scipy's k-means, torch's SDPA) or a
worked example under tests/golden/, so that a dropped term, a wrong sign or
index, or a transposed operand in the oracle fails here.
"""
import numpy as np
import pytest

import oracle
import synth
from conftest import golden

D = 128


def bf16(x):
    return synth.f32_to_bf16_bits(np.asarray(x, np.float32))


def f32(b):
    return synth.bf16_bits_to_f32(b)


# ------------------------------------------------------------------ number formats


def test_fp16_rounding_matches_numpy_and_brackets():
    rng = np.random.default_rng(1)
    xs = np.concatenate([rng.standard_normal(2000) * 10, rng.standard_normal(500) * 1e-5,
                         [0.0, 1.0, -2.5, 65504.0, 6.1e-5, 3e-8]])
    for x in xs:
        near = oracle.round_fp16(x, 0)
        assert near == float(np.float16(x)), x        # numpy's fp16 conversion is round-to-nearest-even
        lo, hi = oracle.round_fp16(x, -1), oracle.round_fp16(x, +1)
        assert lo <= x <= hi
        assert float(np.float16(lo)) == lo and float(np.float16(hi)) == hi
        if lo != hi:
            assert np.nextafter(np.float16(lo), np.float16(np.inf)) == np.float16(hi)
        else:
            assert lo == x


def test_bf16_rne_matches_float32_path():
    rng = np.random.default_rng(2)
    xs = rng.standard_normal(3000).astype(np.float32)  # float32 inputs: no double rounding
    got = np.array([oracle.bf16_rne(float(x)) for x in xs], np.uint16)
    assert np.array_equal(got, bf16(xs))


# ------------------------------------------------------------------ step 1: statistics


def test_stats_expected_logit_perturbation_brute_force():
    """E_Q[(q^T e)^2] = e^T M_h e with M_h = (1/N) sum q q^T (QuantWM, second-order Query statistics)."""
    q = synth.queries(synth.TINY, -1, 256)[0]
    S = np.zeros((D, D))
    oracle.stats_accumulate(q, S)
    M = S / q.shape[0]
    qf = f32(q).astype(np.float64)
    rng = np.random.default_rng(3)
    for _ in range(5):
        e = rng.standard_normal(D)
        brute = np.mean((qf @ e) ** 2)
        assert abs(e @ M @ e - brute) <= 1e-12 * brute


def test_stats_incremental_equals_one_shot():
    q = synth.queries(synth.TINY, 0, 200)[1]
    S1 = np.zeros((D, D)); S2 = np.zeros((D, D))
    oracle.stats_accumulate(q, S1)
    oracle.stats_accumulate(q[:77], S2)
    oracle.stats_accumulate(q[77:], S2)
    np.testing.assert_allclose(S1, S2, rtol=1e-13, atol=0)
    assert np.allclose(S1, S1.T)


def test_weights_diagonal_and_cold_start():
    q = synth.queries(synth.TINY, -1, 64)[0]
    S = np.zeros((D, D))
    oracle.stats_accumulate(q, S)
    w = oracle.weights(S, 64)
    qf = f32(q).astype(np.float64)
    np.testing.assert_allclose(w, np.mean(qf * qf, axis=0), rtol=1e-12)
    assert np.all(oracle.weights(np.zeros((D, D)), 0) == 1.0)


def test_eig_against_numpy_eigh():
    q = synth.queries(synth.TINY, -1, 256)[1]
    S = np.zeros((D, D))
    oracle.stats_accumulate(q, S)
    M = S / 256
    lam, U, sweeps = oracle.eig(M)
    assert sweeps > 0
    ref = np.linalg.eigh(M)[0][::-1]
    np.testing.assert_allclose(lam, ref, rtol=0, atol=1e-12 * np.abs(ref).max())
    assert np.all(np.diff(lam) <= 0)
    assert np.linalg.norm(M @ U - U * lam) <= 1e-12 * np.linalg.norm(M)
    assert np.linalg.norm(U.T @ U - np.eye(D)) <= 1e-12
    # sign convention: the largest-magnitude component of each eigenvector is positive
    arg = np.argmax(np.abs(U), axis=0)
    assert np.all(U[arg, np.arange(D)] > 0)
    # top eigenvectors agree with eigh's up to sign (well separated)
    Ue = np.linalg.eigh(M)[1][:, ::-1]
    for kk in range(8):
        assert abs(abs(U[:, kk] @ Ue[:, kk]) - 1) < 1e-10


def test_eig_diagonal_and_degenerate():
    lam, U, _ = oracle.eig(np.diag([1.0, 3.0, 2.0, 3.0]))
    assert list(lam) == [3.0, 3.0, 2.0, 1.0]
    # ties go to the lower original index: e1 before e3
    assert U[1, 0] == 1.0 and U[3, 1] == 1.0


def test_eig_rank_one_and_two_closed_form():
    """M = q q^T has the single nonzero eigenvalue |q|^2 with eigenvector q / |q|; M = a a^T + b b^T
    with a, b orthogonal has |a|^2, |b|^2 with a / |a|, b / |b|.  The sign convention makes the
    largest-magnitude component positive; every other eigenvalue is 0."""
    rng = np.random.default_rng(11)
    q = rng.standard_normal(D)
    lam, U, _ = oracle.eig(np.outer(q, q))
    assert abs(lam[0] - q @ q) <= 1e-12 * (q @ q)
    assert np.abs(lam[1:]).max() <= 1e-12 * (q @ q)
    u = q / np.linalg.norm(q)
    u = u if u[np.argmax(np.abs(u))] > 0 else -u
    assert np.abs(U[:, 0] - u).max() <= 1e-10
    a = rng.standard_normal(D)
    b = rng.standard_normal(D)
    b -= (a @ b) / (a @ a) * a
    a *= 3.0
    lam, U, _ = oracle.eig(np.outer(a, a) + np.outer(b, b))
    assert abs(lam[0] - a @ a) <= 1e-10 * (a @ a) and abs(lam[1] - b @ b) <= 1e-10 * (a @ a)
    for k, v in ((0, a), (1, b)):
        v = v / np.linalg.norm(v)
        v = v if v[np.argmax(np.abs(v))] > 0 else -v
        assert np.abs(U[:, k] - v).max() <= 1e-9
    # the eigenvectors are orthonormal and the remaining eigenvalues vanish
    assert np.abs(U.T @ U - np.eye(D)).max() <= 1e-10
    assert np.abs(lam[2:]).max() <= 1e-10 * (a @ a)


def test_generator_top8_energy():
    """The Query recipe puts (19.34 + 8 * 0.09) / (19.34 + 128 * 0.09) = 0.65 of the energy in the
    top-8 directions (QuantWM reports more than 60%)."""
    q = synth.queries(synth.P480, 0, 20000)[:2]
    for h in range(2):
        S = np.zeros((D, D))
        oracle.stats_accumulate(q[h], S)
        lam, _, _ = oracle.eig(S / 20000)
        frac = lam[:8].sum() / lam.sum()
        assert 0.60 < frac < 0.70, frac


def test_basis_bf16_rounding():
    U = np.linalg.qr(np.random.default_rng(4).standard_normal((D, D)))[0]
    ur = oracle.basis_bf16(U, 8)
    assert ur.shape == (D, 8)
    assert np.array_equal(ur, bf16(U[:, :8].astype(np.float32)))


# ------------------------------------------------------------------ step 2a: k-means


def test_kmeans_matches_scipy_lloyd():
    vq = pytest.importorskip("scipy.cluster.vq")
    k = synth.keys(synth.TINY)[0]
    x = f32(k).astype(np.float64)
    C, iters = 64, 6
    init = k[(np.arange(C) * k.shape[0]) // C]
    cent, cent64, asg, obj = oracle.kmeans(k, C, None, iters)
    ref, lab = vq.kmeans2(x, f32(init).astype(np.float64), iter=iters, minit="matrix", missing="warn")
    np.testing.assert_allclose(cent64, ref, rtol=1e-12, atol=1e-12)
    assert np.array_equal(cent, bf16(ref.astype(np.float32))) or \
        np.max(np.abs(f32(cent) - ref)) <= np.max(np.abs(ref)) * 2 ** -8
    # Lloyd never increases the objective
    assert np.all(np.diff(obj) <= 1e-9 * obj[0])


def test_kmeans_warm_start_and_objective():
    k = synth.keys(synth.TINY)[1]
    cent, _, asg, obj = oracle.kmeans(k, 32, None, 4)
    # warm start continues the iteration: 4 + 3 iterations from the same start == 7 in one go
    # (up to the bf16 rounding of the hand-over, checked through the objective)
    cent7, _, _, obj7 = oracle.kmeans(k, 32, None, 7)
    cent_w, _, _, obj_w = oracle.kmeans(k, 32, cent, 3)
    assert abs(oracle.kmeans_objective(k, cent_w) - oracle.kmeans_objective(k, cent7)) <= \
        1e-3 * oracle.kmeans_objective(k, cent7)
    # the objective helper equals the brute-force nearest distance sum
    x = f32(k).astype(np.float64)
    mu = f32(cent).astype(np.float64)
    dist = ((x[:, None, :] - mu[None]) ** 2).sum(-1)
    assert abs(oracle.kmeans_objective(k, cent) - dist.min(1).sum()) <= 1e-9 * dist.min(1).sum()


def test_kmeans_one_centroid_per_token_is_exact():
    k = synth.keys(synth.TINY)[0][:40]
    cent, _, asg, obj = oracle.kmeans(k, 40, None, 2)
    assert np.array_equal(cent, k) and obj[-1] == 0.0 and np.array_equal(asg, np.arange(40))


# ------------------------------------------------------------------ step 2: QSAC


def _worked_centroids():
    mu = np.zeros((4, D), np.float32)
    mu[0, 0], mu[0, 1] = 1.0, -1.0
    mu[1, 0] = 1.5
    mu[2, 0] = 10.0
    mu[3, 64], mu[3, 65] = 0.5, -0.5
    return bf16(mu)


def test_qsac_worked_example_golden():
    mu = _worked_centroids()
    k = bf16(np.zeros((1, D), np.float32))
    for row in golden("qsac_worked_example.txt"):
        w = np.ones(D)
        if row["case"] == "B":
            w[64:] = 10.0
        o = oracle.quantize_head(k, k, mu, mu, w, None, top_m=int(row["M"]))
        assert o["idx_k"][0] == int(row["idx"]), row


def test_qsac_uniform_m1_is_nearest_centroid():
    kk = synth.keys(synth.TINY)[0]
    cent, _, _, _ = oracle.kmeans(kk, 256, None, 3)
    o = oracle.quantize_head(kk, kk, cent, cent, None, None, top_m=1)
    x = f32(kk).astype(np.float64)
    mu = f32(cent).astype(np.float64)
    dist = ((x[:, None, :] - mu[None]) ** 2).sum(-1)
    assert np.array_equal(o["idx_k"], dist.argmin(1))
    assert np.array_equal(o["idx_v"], dist.argmin(1))       # Values: nearest centroid


def test_qsac_candidates_are_weighted_nearest_and_choice_is_among_them():
    kk = synth.keys(synth.TINY)[1]
    cent, _, _, _ = oracle.kmeans(kk, 256, None, 3)
    w = np.random.default_rng(5).uniform(0.2, 3.0, D)
    o = oracle.quantize_head(kk, kk, cent, cent, w, None, top_m=4)
    x = f32(kk).astype(np.float64)
    mu = f32(cent).astype(np.float64)
    dq = (w * (x[:, None, :] - mu[None]) ** 2).sum(-1)
    ref = np.argsort(dq, axis=1, kind="stable")[:, :4]
    assert np.array_equal(o["cand"], ref)
    assert all(o["idx_k"][i] in o["cand"][i] for i in range(len(kk)))
    # scaling w by a positive constant changes no decision
    o2 = oracle.quantize_head(kk, kk, cent, cent, w * 7.5, None, top_m=4)
    assert np.array_equal(o["idx_k"], o2["idx_k"])


def test_qsac_exhaustive_candidates_minimise_range_score():
    """With M = C_n every centroid is a candidate: the choice minimises S over all of them.
    The ranges are taken by numpy's max/min on float32 residuals."""
    kk = synth.keys(synth.TINY)[0][:128]
    cent, _, _, _ = oracle.kmeans(synth.keys(synth.TINY)[0], 16, None, 2)
    w = np.random.default_rng(6).uniform(0.5, 2.0, D)
    o = oracle.quantize_head(kk, kk, cent, cent, w, None, top_m=16)
    r = f32(kk)[:, None, :] - f32(cent)[None]                       # float32, exact
    rg = r.reshape(len(kk), 16, 2, 64)
    R = rg.max(-1).astype(np.float64) - rg.min(-1)
    W = w.reshape(2, 64).sum(-1)
    S = (R ** 2 * W).sum(-1)
    assert np.array_equal(o["idx_k"], S.argmin(1))


# ------------------------------------------------------------------ step 3: INT2


def test_int2_worked_example_golden():
    g = {k: v for row in golden("int2_worked_example.txt") for k, v in row.items()}
    r = (np.arange(64) % 4 - 1.5).astype(np.float32)
    codes, s, m = oracle.int2_encode_group(r)
    assert oracle.fp16_val(m) == float(g["m"]) and oracle.fp16_val(s) == float(g["s"])
    assert list(codes[:4]) == [int(c) for c in g["codes"].split(",")]
    assert oracle.pack2(codes)[0] == int(g["byte"], 16)
    codes, s, m = oracle.int2_encode_group(np.full(64, 0.25, np.float32))
    assert oracle.fp16_val(s) == float(g["const_s"]) and oracle.fp16_val(m) == float(g["const_m"])
    assert not codes.any()


def test_pack2_layout_golden():
    g = {k: v for row in golden("pack2_layout.txt") for k, v in row.items()}
    codes = np.zeros(128, np.uint8)
    codes[:8] = [int(c) for c in g["codes"].split(",")]
    packed = oracle.pack2(codes)
    assert list(packed[:2]) == [int(b, 16) for b in g["bytes"].split(",")]


def _decode(codes, s, m):
    sf = np.float32(oracle.fp16_val(s)); mf = np.float32(oracle.fp16_val(m))
    return mf + sf * codes.astype(np.float32)


def test_int2_error_at_most_half_step():
    rng = np.random.default_rng(7)
    cases = [rng.standard_normal(64).astype(np.float32) * sc for sc in (1e-3, 0.3, 1, 8, 100)]
    cases += [np.full(64, 0.3, np.float32), np.zeros(64, np.float32),
              np.r_[np.zeros(63), 1e-4].astype(np.float32), (rng.standard_normal(64) + 50).astype(np.float32)]
    for r in cases:
        codes, s, m = oracle.int2_encode_group(r)
        assert codes.max() <= 3
        sf = oracle.fp16_val(s)
        assert oracle.fp16_val(m) <= r.min()
        assert sf * 3 >= float(r.max()) - oracle.fp16_val(m)
        err = np.abs(r.astype(np.float64) - _decode(codes, s, m))
        assert np.all(err <= sf / 2 * (1 + 2 ** -20) + 1e-30), (err.max(), sf)


def test_int2_uniform_mse_matches_theory():
    """E[e^2] ~ R^2 / [12 (2^b - 1)^2] = R^2 / 108 for b = 2 and uniform residuals (Widrow)."""
    r = synth.unit_residuals(4000, 64, 1)
    mse, pred = 0.0, 0.0
    for row in r:
        codes, s, m = oracle.int2_encode_group(row)
        mse += np.mean((row - _decode(codes, s, m)) ** 2)
        R = float(row.max() - row.min())
        pred += R * R / 108
    assert abs(mse / pred - 1) < 0.05


def test_int8_encode_bound():
    rng = np.random.default_rng(8)
    for sc in (1e-3, 0.1, 5.0):
        Cf = (rng.standard_normal(8) * sc).astype(np.float32)
        c, s = oracle.int8_encode_token(Cf)
        sf = oracle.fp16_val(s)
        assert sf * 127 >= np.abs(Cf).max() and np.abs(c).max() <= 127
        assert np.all(np.abs(Cf - sf * c) <= sf / 2 * (1 + 2 ** -20))
    c, s = oracle.int8_encode_token(np.zeros(8, np.float32))
    assert s == 0 and not c.any()


# ------------------------------------------------------------------ step 4: PSAC


def _psac_case(rank_basis):
    w_ = synth.TINY
    kk = synth.keys(w_)[0][:256]
    vv = synth.values(w_)[0][:256]
    cent_k, _, _, _ = oracle.kmeans(kk, 32, None, 3)
    cent_v, _, _, _ = oracle.kmeans(vv, 32, None, 3)
    q = synth.queries(w_, -1, 256)[0]
    S = np.zeros((D, D))
    oracle.stats_accumulate(q, S)
    M = S / 256
    lam, U, _ = oracle.eig(M)
    return kk, vv, cent_k, cent_v, M, lam, U


def test_psac_full_rank_unquantised_reconstructs_keys():
    """K_hat = K_hat_0 + C U_r^T with C = (K - K_hat_0) U_r is exact when r = d (QuantWM, PSAC)."""
    kk, vv, ck, cv, M, lam, U = _psac_case(D)
    o = oracle.quantize_head(kk, vv, ck, cv, np.diag(M), None, u_r_f64=U, rank=D)
    ch = dict(o, cent_k=ck, cent_v=cv, rank=0)
    _, _, kh0, _ = oracle.dequantize_head(ch)
    k_rec = kh0 + o["c_real"] @ U.T
    assert np.max(np.abs(k_rec - f32(kk))) <= 1e-12


def test_psac_removes_principal_query_error():
    """Query-weighted error e^T M e drops by exactly sum_{k<=r} lambda_k (u_k^T e)^2."""
    kk, vv, ck, cv, M, lam, U = _psac_case(8)
    r = 8
    o = oracle.quantize_head(kk, vv, ck, cv, np.diag(M), None, u_r_f64=U[:, :r].copy(), rank=r)
    ch = dict(o, cent_k=ck, cent_v=cv, rank=0)
    _, _, kh0, _ = oracle.dequantize_head(ch)
    E = f32(kk) - kh0
    E2 = E - o["c_real"] @ U[:, :r].T
    before = np.einsum("ic,cd,id->i", E, M, E)
    after = np.einsum("ic,cd,id->i", E2, M, E2)
    drop = ((E @ U[:, :r]) ** 2 * lam[:r]).sum(1)
    np.testing.assert_allclose(before - after, drop, rtol=1e-9, atol=1e-12)
    assert np.all(after <= before + 1e-12)


# ------------------------------------------------------------------ step 5: attention and decoder


def test_attend_zero_residual_is_textbook_attention_on_centroids():
    """r = 0 (no PSAC) and s = m = 0: attention over mu_idx equals torch SDPA (float64)."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(9)
    n, Cn, nq = 300, 16, 20
    ck = bf16(rng.standard_normal((Cn, D)))
    cv = bf16(rng.standard_normal((Cn, D)))
    ch = dict(idx_k=rng.integers(0, Cn, n), idx_v=rng.integers(0, Cn, n),
              k_codes=rng.integers(0, 256, (n, 32)), v_codes=rng.integers(0, 256, (n, 32)),
              k_scale=np.zeros((n, 2), np.uint16), k_min=np.zeros((n, 2), np.uint16),
              v_scale=np.zeros((n, 2), np.uint16), v_min=np.zeros((n, 2), np.uint16),
              cent_k=ck, cent_v=cv, rank=0)
    q = bf16(rng.standard_normal((nq, D)) * 2)
    out = oracle.attend_rows(q, np.arange(nq), [ch], 1 / np.sqrt(D))
    Q = torch.tensor(f32(q), dtype=torch.float64)[None]
    K = torch.tensor(f32(ck)[ch["idx_k"]], dtype=torch.float64)[None]
    V = torch.tensor(f32(cv)[ch["idx_v"]], dtype=torch.float64)[None]
    ref = torch.nn.functional.scaled_dot_product_attention(Q, K, V)[0].numpy()
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)


def test_attend_equals_sdpa_on_decoded_cache_with_psac():
    """The logit form Q K_hat_0^T + (Q U_r) C^T equals attention over K_hat = K_hat_0 + C U_r^T,
    across two chunks with different bases."""
    torch = pytest.importorskip("torch")
    w_ = synth.TINY
    kk = synth.keys(w_)[0]; vv = synth.values(w_)[0]
    q = synth.queries(w_, 0, 64)[0]
    chunks, Ks, Vs = [], [], []
    for t, (a, b) in enumerate([(0, 512), (512, 1024)]):
        ck, _, _, _ = oracle.kmeans(kk[a:b], 64, None, 2)
        cv, _, _, _ = oracle.kmeans(vv[a:b], 64, None, 2)
        U = np.linalg.qr(np.random.default_rng(10 + t).standard_normal((D, D)))[0]
        ur = oracle.basis_bf16(U, 8)
        o = oracle.quantize_head(kk[a:b], vv[a:b], ck, cv, None, ur)
        ch = dict(o, cent_k=ck, cent_v=cv, u_r=ur, rank=8)
        chunks.append(ch)
        _, _, kh, vh = oracle.dequantize_head(ch)
        Ks.append(kh); Vs.append(vh)
    out = oracle.attend_rows(q, np.arange(64), chunks, 1 / np.sqrt(D))
    Q = torch.tensor(f32(q), dtype=torch.float64)[None]
    K = torch.tensor(np.concatenate(Ks))[None]
    V = torch.tensor(np.concatenate(Vs))[None]
    ref = torch.nn.functional.scaled_dot_product_attention(Q, K, V)[0].numpy()
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-11)


def test_dequantize_bf16_is_rounded_float64():
    w_ = synth.TINY
    kk = synth.keys(w_)[1][:200]; vv = synth.values(w_)[1][:200]
    ck, _, _, _ = oracle.kmeans(kk, 32, None, 2)
    cv, _, _, _ = oracle.kmeans(vv, 32, None, 2)
    ur = oracle.basis_bf16(np.linalg.qr(np.random.default_rng(11).standard_normal((D, D)))[0], 8)
    o = oracle.quantize_head(kk, vv, ck, cv, None, ur)
    kh, vh, kh64, vh64 = oracle.dequantize_head(dict(o, cent_k=ck, cent_v=cv, u_r=ur, rank=8))
    # float64 -> bf16 directly; float32 inputs round identically, so compare through float32
    # where float32 holds the value exactly and within one bf16 step elsewhere
    for h, h64 in ((kh, kh64), (vh, vh64)):
        assert np.all(np.abs(f32(h) - h64) <= np.abs(h64) * 2 ** -8 + 1e-30)


# ---------------------------------------------------------------- comparison baselines


def _bf(a):
    return (np.asarray(a, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _f16(a):
    return np.asarray(a, np.uint16).view(np.float16).astype(np.float64)


def test_prq_residual_zero_on_own_centroid_and_exact_second_stage():
    """Quant VideoGen §2B: a token that is its own stage-1 centroid leaves a zero residual; a
    stage-2 codebook holding the exact residuals reconstructs every token exactly (INT2 of zero)."""
    k, v, _, _ = synth.small_case(1, 96, 128, 96, 8, seed=41)
    k, v = k[0], v[0]
    idx = np.arange(96)
    assert not oracle.prq_residual(k, k, idx).any()
    # stage 1: 16 centroids (tokens 0, 6, 12, ...); stage 2: each token's own residual
    c1k, c1v = k[::6].copy(), v[::6].copy()
    o1 = oracle.quantize_head(k, v, c1k, c1v, None, None, top_m=1, rank=0)
    r1k = oracle.prq_residual(k, c1k, o1["idx_k"])
    r1v = oracle.prq_residual(v, c1v, o1["idx_v"])
    out = oracle.prq_head(k, v, [c1k, r1k], [c1v, r1v])
    # the residual is rounded to bf16, so the reconstruction is x up to that rounding
    rk = _bf(k) - _bf(c1k)[out["idx_k"][0]]
    assert np.all(np.abs(out["k_hat"] - _bf(k)) <= np.abs(rk) * 2.0 ** -8 + 1e-30)
    assert np.array_equal(out["idx_k"][1], np.arange(96)) or np.all(out["last"]["k_scale"] == 0)


def test_prq_two_stage_error_bound():
    """Decoded tokens of a two-stage chunk: |x - x_hat| <= s/2 (INT2 of the last residual) plus half a
    bf16 step of the rounded stage-1 residual, per element."""
    k, v, _, _ = synth.small_case(1, 300, 128, 64, 8, seed=42)
    k, v = k[0], v[0]
    c1k, _, _, _ = oracle.kmeans(k, 16, None, 3)
    c1v, _, _, _ = oracle.kmeans(v, 16, None, 3)
    o1 = oracle.quantize_head(k, v, c1k, c1v, None, None, top_m=1, rank=0)
    r1 = oracle.prq_residual(k, c1k, o1["idx_k"])
    c2k, _, _, _ = oracle.kmeans(r1, 16, None, 3)
    r1v = oracle.prq_residual(v, c1v, o1["idx_v"])
    c2v, _, _, _ = oracle.kmeans(r1v, 16, None, 3)
    out = oracle.prq_head(k, v, [c1k, c2k], [c1v, c2v])
    s = _f16(out["last"]["k_scale"])[:, np.arange(128) // 64]
    exact_r1 = _bf(k) - _bf(c1k)[out["idx_k"][0]]
    bound = s / 2 + np.abs(exact_r1) * 2.0 ** -8 + 1e-12  # half a bf16 step of r1 is at most |r1| 2^-8
    assert np.all(np.abs(out["k_hat"] - _bf(k)) <= bound)
    assert np.all(out["idx_k"][0] == o1["idx_k"])


def _f16_down(x):
    h = np.float16(x)
    return h if float(h) <= x else np.nextafter(h, np.float16(-np.inf))


def test_kivi_groups_error_bound_and_axes():
    """KIVI-style INT2: Keys grouped per channel over 32 consecutive tokens (ragged last group),
    Values per token over 32 consecutive channels.  Each group's offset is the fp16 round-down of
    that group's minimum (brute force over the right axis), and every element is within s/2."""
    k, v, _, _ = synth.small_case(1, 100, 128, 64, 8, seed=43)
    k, v = k[0], v[0]
    o = oracle.kivi_quantize_head(k, v, 32)
    assert o["k_scale"].shape == (4, 128) and o["v_scale"].shape == (100, 4)
    kf, vf = _bf(k), _bf(v)
    for tg in range(4):
        for c in (0, 5, 127):
            seg = kf[32 * tg:32 * tg + 32, c]
            assert _f16(o["k_min"][tg, c]) == float(_f16_down(seg.min()))
    for t in (0, 50, 99):
        for cg in range(4):
            assert _f16(o["v_min"][t, cg]) == float(_f16_down(vf[t, 32 * cg:32 * cg + 32].min()))
    kh, vh = oracle.kivi_dequantize_head(o, 32)
    sk = _f16(o["k_scale"])[np.arange(100) // 32]
    sv = _f16(o["v_scale"])[:, np.arange(128) // 32]
    assert np.all(np.abs(kh - kf) <= sk / 2 + 1e-12)
    assert np.all(np.abs(vh - vf) <= sv / 2 + 1e-12)


def test_kivi_constant_groups_are_exact():
    """A channel that is constant over a token group (Keys) or a channel group that is constant in a
    token (Values) has s = 0 and decodes exactly."""
    k = np.full((64, 128), synth.f32_to_bf16_bits(np.float32(1.5)), np.uint16)
    v = np.full((64, 128), synth.f32_to_bf16_bits(np.float32(-0.25)), np.uint16)
    o = oracle.kivi_quantize_head(k, v, 32)
    assert not o["k_scale"].any() and not o["v_scale"].any()
    kh, vh = oracle.kivi_dequantize_head(o, 32)
    assert np.all(kh == 1.5) and np.all(vh == -0.25)


# ---------------------------------------------------------------- the chunk still being generated (bf16)


def _np_attention(q, k, v, scale, mask=None):
    L = (q @ k.T) * scale
    if mask is not None:
        L = np.where(mask, L, -np.inf)
    P = np.exp(L - L.max(1, keepdims=True))
    return (P / P.sum(1, keepdims=True)) @ v


def test_attend_bf16_chunk_is_textbook_attention():
    k, v, _, qa = synth.small_case(1, 200, 128, 64, 40, seed=51)
    raw = dict(k_raw=k[0], v_raw=v[0])
    out = oracle.attend_rows(qa[0], np.arange(40), [raw], 0.09)
    ref = _np_attention(_bf(qa[0]), _bf(k[0]), _bf(v[0]), 0.09)
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-12)


def test_attend_block_causal_mask():
    """Frames of tpf tokens: row q sees key j only when j // tpf <= q // tpf.  Brute-force mask;
    tpf = 1 makes row 0 attend to key 0 alone (its output is v_0 exactly); tpf = n removes the mask."""
    n = 96
    k, v, _, _ = synth.small_case(1, n, 128, 32, 8, seed=52)
    q = synth.small_case(1, n, 128, 32, n, seed=53)[3][0]
    rows = np.arange(n)
    for tpf in (32, 7):
        raw = dict(k_raw=k[0], v_raw=v[0], causal_tpf=tpf)
        mask = (np.arange(n)[None, :] // tpf) <= (rows[:, None] // tpf)
        out = oracle.attend_rows(q, rows, [raw], 0.1)
        assert np.allclose(out, _np_attention(_bf(q), _bf(k[0]), _bf(v[0]), 0.1, mask), rtol=1e-12, atol=1e-12)
    out1 = oracle.attend_rows(q, rows[:1], [dict(k_raw=k[0], v_raw=v[0], causal_tpf=1)], 0.1)
    assert np.array_equal(out1[0], _bf(v[0])[0])
    outn = oracle.attend_rows(q, rows, [dict(k_raw=k[0], v_raw=v[0], causal_tpf=n)], 0.1)
    assert np.allclose(outn, oracle.attend_rows(q, rows, [dict(k_raw=k[0], v_raw=v[0])], 0.1), rtol=0, atol=0)


def test_attend_packed_and_bf16_chunks_share_one_softmax():
    """A packed chunk followed by a bf16 chunk: one softmax over the decoded packed keys and the raw
    keys together."""
    k, v, qs, qa = synth.small_case(1, 300, 128, 64, 24, seed=54)
    ck, _, _, _ = oracle.kmeans(k[0, :200], 64, None, 3)
    cv, _, _, _ = oracle.kmeans(v[0, :200], 64, None, 3)
    o = oracle.quantize_head(k[0, :200], v[0, :200], ck, cv, None, None, top_m=1, rank=0)
    packed = dict(idx_k=o["idx_k"], idx_v=o["idx_v"], k_codes=o["k_codes"], v_codes=o["v_codes"],
                  k_scale=o["k_scale"], k_min=o["k_min"], v_scale=o["v_scale"], v_min=o["v_min"],
                  cent_k=ck, cent_v=cv, rank=0)
    _, _, kh, vh = oracle.dequantize_head(packed)
    raw = dict(k_raw=k[0, 200:], v_raw=v[0, 200:])
    out = oracle.attend_rows(qa[0], np.arange(24), [packed, raw], 0.08)
    ref = _np_attention(_bf(qa[0]), np.concatenate([kh, _bf(k[0, 200:])]), np.concatenate([vh, _bf(v[0, 200:])]), 0.08)
    assert np.allclose(out, ref, rtol=1e-10, atol=1e-12)


def test_attend_log_sum_exp_and_merge_identity():
    """The rows' base-2 log-sum-exp of the logits equals scipy's logsumexp / ln 2 on textbook logits
    (raw bf16 keys); and the softmax over a union of chunks is the mean of the parts' softmaxes
    weighted by 2^(lse_part - lse_union), lse_union = log2(2^lse_A + 2^lse_B) -- the identity the GPU's
    merging attention relies on -- with a packed and a bf16 chunk as the parts."""
    special = pytest.importorskip("scipy.special")
    k, v, _, qa = synth.small_case(1, 200, 128, 64, 40, seed=55)
    raw = dict(k_raw=k[0], v_raw=v[0])
    _, lse = oracle.attend_rows(qa[0], np.arange(40), [raw], 0.09, with_lse=True)
    logits = (_bf(qa[0]) @ _bf(k[0]).T) * 0.09
    assert np.allclose(lse, special.logsumexp(logits, axis=1) / np.log(2.0), rtol=1e-13, atol=1e-12)
    k, v, _, qa = synth.small_case(1, 300, 128, 64, 24, seed=54)
    ck, _, _, _ = oracle.kmeans(k[0, :200], 64, None, 3)
    cv, _, _, _ = oracle.kmeans(v[0, :200], 64, None, 3)
    o = oracle.quantize_head(k[0, :200], v[0, :200], ck, cv, None, None, top_m=1, rank=0)
    packed = dict(idx_k=o["idx_k"], idx_v=o["idx_v"], k_codes=o["k_codes"], v_codes=o["v_codes"],
                  k_scale=o["k_scale"], k_min=o["k_min"], v_scale=o["v_scale"], v_min=o["v_min"],
                  cent_k=ck, cent_v=cv, rank=0)
    raw = dict(k_raw=k[0, 200:], v_raw=v[0, 200:])
    rows = np.arange(24)
    oa, la = oracle.attend_rows(qa[0], rows, [packed], 0.08, with_lse=True)
    ob, lb = oracle.attend_rows(qa[0], rows, [raw], 0.08, with_lse=True)
    ou, lu = oracle.attend_rows(qa[0], rows, [packed, raw], 0.08, with_lse=True)
    assert np.allclose(lu, np.logaddexp2(la, lb), rtol=1e-13, atol=1e-12)
    wa, wb = np.exp2(la - lu)[:, None], np.exp2(lb - lu)[:, None]
    assert np.allclose(ou, wa * oa + wb * ob, rtol=1e-10, atol=1e-12)


# ---------------------------------------------------------------- compact metadata and the PSAC gate


def _codes(packed):
    n, d4 = packed.shape
    out = np.zeros((n, 4 * d4), np.int64)
    for c in range(4 * d4):
        out[:, c] = (packed[:, c // 4] >> (2 * (c % 4))) & 3
    return out


def test_compact_metadata_bound_and_grid():
    """Compact metadata (step (3): INT8 group scale + fp16 second-level scale; §D.1: INT2 zero-points):
    r_hat = sigma s8 (q - z) reproduces every residual within s/2; sigma is a power of two per 128-token
    tile and group, minimal for the tile's largest step (so that step's s8 lies in [128, 255]); a group
    whose residuals are all >= 0 takes z = 0, all <= 0 takes z = 3; no zero-point gives a smaller step."""
    k, v, _, _ = synth.small_case(1, 300, 128, 64, 8, seed=61)
    k, v = k[0], v[0]
    ck, _, _, _ = oracle.kmeans(k, 32, None, 3)
    cv, _, _, _ = oracle.kmeans(v, 32, None, 3)
    o = oracle.quantize_head(k, v, ck, cv, None, None, top_m=1, rank=0, storage=1)
    for pre, x, cent in (("k", k, ck), ("v", v, cv)):
        idx = o["idx_" + pre]
        r = (_bf(x) - _bf(cent)[idx]).astype(np.float32).astype(np.float64)
        sig = _f16(o[pre + "_sigma"])                      # [tiles][2]
        s8 = o[pre + "_s8"].astype(np.float64)             # [n][2]
        z = np.stack([(o[pre + "_zp"] >> (2 * g)) & 3 for g in range(2)], 1).astype(np.float64)
        s = sig[np.arange(300) // 128] * s8
        q = _codes(o[pre + "_codes"])
        g = np.arange(128) // 64
        rh = s[:, g] * (q - z[:, g])
        assert np.all(np.abs(r - rh) <= s[:, g] / 2 + 1e-12)
        nz = sig > 0
        assert np.all(np.log2(sig[nz]) == np.round(np.log2(sig[nz])))
        for t in range(3):
            for gg in range(2):
                rows = slice(128 * t, min(300, 128 * t + 128))
                if sig[t, gg] > 0:
                    assert 128 <= s8[rows, gg].max() <= 255
        for i in range(0, 300, 7):
            for gg in range(2):
                a, b = r[i, 64 * gg:64 * gg + 64].min(), r[i, 64 * gg:64 * gg + 64].max()
                if a >= 0 and b > 0:
                    assert z[i, gg] == 0
                if b <= 0 and a < 0:
                    assert z[i, gg] == 3
                # the smallest covering step over the four zero-points never exceeds the chosen one
                need = min(max(-a / zz if zz else (0 if a >= 0 else np.inf), b / (3 - zz) if zz < 3 else (0 if b <= 0 else np.inf))
                           for zz in range(4))
                assert need <= s[i, gg] * (1 + 1e-6) + 1e-30


def test_psac_gate_keeps_only_improving_coefficients():
    """Step (4): C is kept only when it lowers the Query-weighted error.  With heavily uneven
    weights some tokens' coefficients must be dropped; every dropped token has e1 >= e0 and every
    kept one e1 < e0, recomputed here from the decoded K_hat_0 and C_hat."""
    k, v, qs, _ = synth.small_case(1, 400, 128, 64, 256, seed=62)
    S = np.zeros((1, 128, 128)); nn = np.zeros(1, np.int64)
    w, _, ur, _, _ = oracle.update_query_stats(qs, S, nn, 8)
    w = w[0].copy()
    w[::3] *= 50.0                                          # uneven channel weights
    ck, _, _, _ = oracle.kmeans(k[0], 64, None, 3)
    cv, _, _, _ = oracle.kmeans(v[0], 64, None, 3)
    base = oracle.quantize_head(k[0], v[0], ck, cv, w, ur[0], top_m=4, rank=8)
    gated = oracle.quantize_head(k[0], v[0], ck, cv, w, ur[0], top_m=4, rank=8, psac_gate=1)
    ch = dict(idx_k=base["idx_k"], idx_v=base["idx_v"], k_codes=base["k_codes"], v_codes=base["v_codes"],
              k_scale=base["k_scale"], k_min=base["k_min"], v_scale=base["v_scale"], v_min=base["v_min"],
              cent_k=ck, cent_v=cv, rank=0)
    _, _, kh0, _ = oracle.dequantize_head(ch)
    E = _bf(k[0]) - kh0
    corr = (_f16(base["c_scale"])[:, None] * base["c"].astype(np.float64)) @ _bf(ur[0]).T
    e0 = (w * E * E).sum(1)
    e1 = (w * (E - corr) ** 2).sum(1)
    drop = ~(e1 < e0)
    assert drop.any() and (~drop).any()
    assert np.all(gated["c"][drop] == 0) and np.all(gated["c_scale"][drop] == 0)
    assert np.array_equal(gated["c"][~drop], base["c"][~drop])
    assert np.array_equal(gated["c_scale"][~drop], base["c_scale"][~drop])


# ---------------------------------------------------------------- full quadratic-form ranking (§C.4 ablation)


def test_full_form_ranking_reduces_to_diagonal_and_matches_brute_force():
    """English v2 §C.4: the ablation ranks candidates by (k - mu)^T M (k - mu).  With M diagonal it is
    the diagonal QSAC exactly; with a general PSD M the candidates are the M smallest quadratic forms
    (brute force with numpy), and the choice among them is still the range score with w = diag(M)."""
    k, v, qs, _ = synth.small_case(1, 120, 128, 64, 200, seed=71)
    k, v = k[0], v[0]
    ck, _, _, _ = oracle.kmeans(k, 64, None, 3)
    cv, _, _, _ = oracle.kmeans(v, 64, None, 3)
    w = np.linspace(0.5, 2.0, 128)
    diag = oracle.quantize_head(k, v, ck, cv, w, None, top_m=4, rank=0)
    full_diag = oracle.quantize_head(k, v, ck, cv, w, None, top_m=4, rank=0, M_full=np.diag(w))
    assert np.array_equal(diag["idx_k"], full_diag["idx_k"])
    assert np.array_equal(np.sort(diag["cand"], 1), np.sort(full_diag["cand"], 1))
    q = _bf(qs[0])
    M = q.T @ q / q.shape[0]
    o = oracle.quantize_head(k, v, ck, cv, np.diag(M).copy(), None, top_m=4, rank=0, M_full=M)
    E = _bf(k)[:, None, :] - _bf(ck)[None, :, :]
    dq = np.einsum("ijc,cd,ijd->ij", E, M, E)
    srt = np.sort(dq, 1)
    clear = (srt[:, 4] - srt[:, 3]) > 1e-9 * srt[:, 3]
    ref = np.sort(np.argsort(dq, 1, kind="stable")[:, :4], 1)
    assert np.array_equal(np.sort(o["cand"], 1)[clear], ref[clear])
    assert np.all([o["idx_k"][i] in o["cand"][i] for i in range(120)])


# ---------------------------------------------------------------- PSAC rank per head and coefficient layouts


def test_adaptive_rank_closed_form_spectra():
    """The smallest r whose top-r eigenvalues hold a share of tr M, on spectra whose cumulative
    shares are known in closed form."""
    geo = 2.0 ** -np.arange(128)                            # share after r: (1 - 2^-r) / (1 - 2^-128)
    assert oracle.adaptive_rank(geo, 16, 0.9) == 4          # 0.875 < 0.9 <= 0.9375
    assert oracle.adaptive_rank(geo, 16, 0.5) == 1
    assert oracle.adaptive_rank(geo, 3, 0.99) == 3          # capped at r_max
    flat = np.ones(128)                                     # share after r: r / 128
    assert oracle.adaptive_rank(flat, 16, 10 / 128) == 10
    assert oracle.adaptive_rank(flat, 16, 0.5) == 16        # 64 needed, capped
    one = np.zeros(128); one[17] = 5.0                      # rank one (order of input irrelevant)
    assert oracle.adaptive_rank(one, 8, 1.0) == 1
    assert oracle.adaptive_rank(np.zeros(128), 8, 0.5) == 0  # no Query seen
    assert oracle.adaptive_rank(geo, 8, 0.0) == 0


def test_adaptive_rank_brute_force():
    rng = np.random.default_rng(71)
    for _ in range(200):
        lam = np.sort(rng.gamma(0.5, 1.0, 128))[::-1]
        tau, rmax = rng.uniform(0, 1), int(rng.integers(0, 17))
        share = np.concatenate([[0.0], np.cumsum(lam)]) / lam.sum()
        ok = [r for r in range(rmax + 1) if share[r] >= tau - 1e-12]
        assert oracle.adaptive_rank(lam, rmax, tau) == (ok[0] if ok else rmax)


@pytest.mark.parametrize("n,frac", [(300, 0.3), (1000, 1.0), (257, 0.0), (10800, 0.9)])
def test_psac_sparse_layout_round_trip(n, frac):
    """The sparse layout decodes to the dense one exactly: every kept token (non-zero scale) finds
    its row through the bitmap and the per-tile counts; a dropped token decodes to zeros."""
    rng = np.random.default_rng(n)
    r = 8
    c = rng.integers(-127, 128, size=(n, r)).astype(np.int8)
    sc = rng.integers(1, 0x7BFF, size=n).astype(np.uint16)
    drop = rng.random(n) >= frac
    sc[drop] = 0
    c[drop] = 0                                             # what the gate stores for a dropped token
    mask, tile_rank, rows, scales = oracle.psac_sparse_encode(c, sc)
    assert rows.shape == ((~drop).sum(), r)
    pop = np.array([sum(bin(int(x)).count("1") for x in m) for m in mask])
    assert pop.sum() == (~drop).sum()
    assert np.array_equal(tile_rank, np.concatenate([[0], np.cumsum(pop)[:-1]]).astype(np.int32))
    c2, sc2 = oracle.psac_sparse_decode(mask, tile_rank, rows, scales, n, r)
    assert np.array_equal(c2, c) and np.array_equal(sc2, sc)


def test_psac_layout_choice_is_the_smaller():
    n, r = 10800, 8
    tiles = (n + 127) // 128
    for kept in (0, 5000, 10629, 10630, 10631, n):
        dense, sparse = oracle.psac_layout_bytes(n, r, kept)
        assert dense == n * 10 and sparse == kept * 10 + tiles * 20
        (use_sparse, rows), = oracle.psac_plan(n, [r], [kept])
        assert use_sparse == (kept * 10 + 1700 < 108000) and rows == (kept if use_sparse else n)
    assert oracle.psac_plan(n, [0], [0]) == [(False, 0)]     # a head without PSAC stores nothing


def test_psac_gate_drops_every_token_when_the_basis_sees_only_unweighted_channels():
    """With zero weight on channels 64..127 and a basis supported there, the correction never
    changes the Query-weighted error, so the gate (strict improvement) drops every token and the
    sparse layout stores no row; moving part of the basis onto weighted channels keeps some."""
    k, v, qs, _ = synth.small_case(1, 300, 128, 64, 256, seed=72)
    ck, _, _, _ = oracle.kmeans(k[0], 64, None, 3)
    cv, _, _, _ = oracle.kmeans(v[0], 64, None, 3)
    w = np.r_[np.ones(64), np.zeros(64)]
    U = np.zeros((128, 8)); U[64 + np.arange(8) * 8, np.arange(8)] = 1.0
    o = oracle.quantize_head(k[0], v[0], ck, cv, w, bf16(U), top_m=4, rank=8, psac_gate=1)
    assert np.all(o["c_scale"] == 0) and np.all(o["c"] == 0)
    (use_sparse, rows), = oracle.psac_plan(300, [8], [0])
    assert use_sparse and rows == 0
    U2 = U.copy(); U2[np.arange(8) * 8, np.arange(8)] = 0.5
    U2 /= np.linalg.norm(U2, axis=0)
    o2 = oracle.quantize_head(k[0], v[0], ck, cv, w, bf16(U2), top_m=4, rank=8, psac_gate=1)
    kept = int((o2["c_scale"] != 0).sum())
    assert 0 < kept <= 300


def test_codebook_fp16_is_round_to_nearest_of_the_bf16_values():
    """The stored codebook is the fp16 value of each bf16 centroid element: numpy's float16
    conversion (round to nearest even), exact for magnitudes in [2^-17, 65504] and for 0."""
    rng = np.random.default_rng(81)
    x = np.concatenate([rng.standard_normal(2000), rng.standard_normal(200) * 2.0 ** -16,
                        rng.standard_normal(100) * 2.0 ** -20, [0.0, -0.0, 65504.0, 1e5, 2.0 ** -17, 3 * 2.0 ** -19]])
    b = bf16(x)
    got = oracle.codebook_fp16(b)
    with np.errstate(over="ignore"):                        # 1e5 overflows to inf, as in the oracle
        want = f32(b).astype(np.float16).view(np.uint16)
    assert np.array_equal(got, want)
    v = f32(b).astype(np.float64)
    exact = (np.abs(v) >= 2.0 ** -17) & (np.abs(v) <= 65504.0) | (v == 0)
    assert np.all(want[exact].view(np.float16).astype(np.float64) == v[exact])


def test_decode_from_stored_fp16_codebook():
    """Decoding with the stored fp16 codebook equals decoding with the bf16 one when every element is
    exact in fp16; an element below 2^-17 decodes through its fp16 rounding."""
    k, v, qs, _ = synth.small_case(1, 200, 128, 64, 64, seed=82)
    ck, _, _, _ = oracle.kmeans(k[0], 64, None, 3)
    cv, _, _, _ = oracle.kmeans(v[0], 64, None, 3)
    ckv = f32(ck).astype(np.float64)
    ck = np.where((np.abs(ckv) < 2.0 ** -17) & (ckv != 0), bf16(np.full(ck.shape, 0.5)), ck)  # all exact
    o = oracle.quantize_head(k[0], v[0], ck, cv, None, None, top_m=4)
    base = dict(idx_k=o["idx_k"], idx_v=o["idx_v"], k_codes=o["k_codes"], v_codes=o["v_codes"],
                k_scale=o["k_scale"], k_min=o["k_min"], v_scale=o["v_scale"], v_min=o["v_min"], rank=0)
    a = oracle.dequantize_head(dict(base, cent_k=ck, cent_v=cv))
    b = oracle.dequantize_head(dict(base, cent_k16=oracle.codebook_fp16(ck), cent_v16=oracle.codebook_fp16(cv)))
    for x, y in zip(a, b):
        assert np.array_equal(x, y)
    tiny = ck.copy()
    j = int(o["idx_k"][0])
    tiny[j, 5] = bf16([3.3e-6])[0]                          # below 2^-17: rounds in fp16
    c16 = oracle.codebook_fp16(tiny)
    _, _, k64, _ = oracle.dequantize_head(dict(base, cent_k16=c16, cent_v16=oracle.codebook_fp16(cv)))
    _, _, k64b, _ = oracle.dequantize_head(dict(base, cent_k=tiny, cent_v=cv))
    d = k64[0, 5] - k64b[0, 5]
    assert d == np.float16(f32(tiny[j, 5])).astype(np.float64) - f32(tiny[j, 5]).astype(np.float64) and d != 0
