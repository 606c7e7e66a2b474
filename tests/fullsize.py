"""Full-size parity helpers (tests only): stream one synthetic layer through the CUDA path chunk by
chunk, then let the oracle recompute sampled outputs one by one from the GPU's upstream state
(statistics, codebooks, basis, the packed chunks)."""
import math

import numpy as np

import oracle
import synth
from helpers import bf16_ulp_close, chunk_head, decode_term_magnitude, from_u16, to_u16

D = 128
TIE = 1e-5


def stream_layer(W, layer: int = 0, **ctx_kwargs):
    """Stream all chunks of `layer` of workload W: fold the previous chunk's Queries, fit and pack the
    chunk (stage outputs of the last chunk kept), and attend the last chunk's Queries over every
    packed chunk."""
    import torch

    import bit_kv_cache_qsac_gb300 as q
    from bit_kv_cache_qsac_gb300.stream import CompressedLayer
    ctx = q.Context(heads=W.heads, **ctx_kwargs)
    cfg = ctx.cfg
    lay = CompressedLayer(ctx, keep_fit_codebooks=True)
    ks, vs, qs = [], [], []
    for t in range(W.n_chunks):
        a, b = synth.chunk_range(W, t)
        ks.append(synth.keys(W, layer, a, b)); vs.append(synth.values(W, layer, a, b))
        qs.append(synth.queries(W, t, W.nq_attend, layer))
    dbg = None
    for t in range(W.n_chunks):
        if t > 0:
            lay.fold_queries(from_u16(qs[t - 1], torch.bfloat16))
        if t == W.n_chunks - 1 and cfg.rank > 0:
            n = W.chunk_tokens
            dbg = dict(c_f32=torch.zeros(W.heads, n, cfg.rank, device="cuda"),
                       cand=torch.zeros(W.heads, n, cfg.top_m, dtype=torch.int32, device="cuda"))
        lay.append_chunk(from_u16(ks[t], torch.bfloat16), from_u16(vs[t], torch.bfloat16), debug=dbg)
    out = lay.attend(from_u16(qs[-1], torch.bfloat16))
    torch.cuda.synchronize()
    assert lay.check() == 0
    return dict(q=q, W=W, cfg=cfg, layer=lay, ks=ks, vs=vs, qs=qs, out=out, dbg=dbg)


def check_statistics(run, heads):
    W, lay, qs = run["W"], run["layer"], run["qs"]
    for h in heads:
        S = np.zeros((D, D))
        for t in range(W.n_chunks - 1):
            oracle.stats_accumulate(qs[t][h], S)
        assert int(lay.n[h]) == (W.n_chunks - 1) * W.nq_attend
        np.testing.assert_allclose(lay.S[h].cpu().numpy(), S, rtol=1e-4, atol=1e-4 * np.abs(S).max())
        lam, _, _ = oracle.eig(lay.S[h].cpu().numpy().astype(np.float64) / float(lay.n[h]))
        gl = lay.eigvals[h].cpu().numpy()
        assert np.all(np.abs(gl - lam) <= 1e-3 * np.abs(lam) + 1e-6 * lam[0])


def check_kmeans(run, h, tensor="k"):
    lay, xs, cfg = run["layer"], run["ks" if tensor == "k" else "vs"], run["cfg"]
    name = "cent_" + tensor
    init = to_u16(getattr(lay.chunks[-2], name)[h])
    ref, _, _, _ = oracle.kmeans(xs[-1][h], cfg.n_centroids, init, cfg.kmeans_iters)
    j_gpu = oracle.kmeans_objective(xs[-1][h], to_u16(getattr(lay.chunks[-1], name)[h]))
    j_ref = oracle.kmeans_objective(xs[-1][h], ref)
    assert abs(j_gpu - j_ref) <= 1e-3 * j_ref, (j_gpu, j_ref)


def check_packing(run, heads, rows):
    """Indices bit-exact outside ties; codes, scales and offsets bit-exact after re-encoding with the
    GPU's indices; C within 1e-3 of the oracle's (relative to the token's largest |C|); INT8 C and
    its scale bit-exact given the GPU's fp32 C.  Returns the tie counts."""
    W, lay, ks, vs, dbg, cfg = run["W"], run["layer"], run["ks"], run["vs"], run["dbg"], run["cfg"]
    ch = lay.chunks[-1]
    ties = np.zeros(3, np.int64)
    for h in heads:
        w = lay.w[h].cpu().numpy().astype(np.float64)
        ur = to_u16(ch.u_r[h])[:, :cfg.rank] if cfg.rank else None
        k, v = ks[-1][h][rows], vs[-1][h][rows]
        o = oracle.quantize_head(k, v, to_u16(ch.cent_k[h]), to_u16(ch.cent_v[h]), w, ur, top_m=cfg.top_m)
        gk = ch.k_idx[h].cpu().numpy()[rows].astype(np.int32)
        gv = ch.v_idx[h].cpu().numpy()[rows].astype(np.int32)
        s2, de, vd = o["score2"], o["dq_edge"], o["vdist2"]
        tie_s = np.abs(s2[:, 1] - s2[:, 0]) <= TIE * np.abs(s2[:, 0])
        tie_e = np.abs(de[:, 1] - de[:, 0]) <= TIE * np.abs(de[:, 0])
        tie_v = np.abs(vd[:, 1] - vd[:, 0]) <= TIE * np.abs(vd[:, 0])
        ties += [tie_s.sum(), tie_e.sum(), tie_v.sum()]
        assert np.all((gk == o["idx_k"]) | tie_s | tie_e), np.nonzero((gk != o["idx_k"]) & ~(tie_s | tie_e))
        assert np.all((gv == o["idx_v"]) | tie_v)
        o2 = oracle.quantize_head(k, v, to_u16(ch.cent_k[h]), to_u16(ch.cent_v[h]), w, ur, top_m=cfg.top_m,
                                  force_idx_k=gk, force_idx_v=gv)
        for name in ("k_codes", "v_codes"):
            assert np.array_equal(getattr(ch, name)[h].cpu().numpy()[rows], o2[name]), name
        for name in ("k_scale", "k_min", "v_scale", "v_min"):
            assert np.array_equal(to_u16(getattr(ch, name)[h])[rows], o2[name]), name
        if cfg.rank:
            cg = dbg["c_f32"][h].cpu().numpy()[rows].astype(np.float64)
            scale_ = np.maximum(np.abs(o2["c_real"]).max(1, keepdims=True), 1e-30)
            assert np.all(np.abs(cg - o2["c_real"]) <= 1e-3 * scale_)
            gc8 = ch.c[h].cpu().numpy()[rows]
            gsc = to_u16(ch.c_scale[h])[rows]
            for i in range(len(rows)):
                c8, sc = oracle.int8_encode_token(cg[i].astype(np.float32))
                assert sc == gsc[i] and np.array_equal(c8, gc8[i])
    return ties


def check_decoder(run, h, chunk=-1):
    lay = run["layer"]
    kh, vh = lay.dequantize(len(lay.chunks) - 1 if chunk == -1 else chunk)
    ch = chunk_head(lay.chunks[chunk], h)
    k32, v32, k64, v64 = oracle.dequantize_head(ch)
    for got, ref, key in ((to_u16(kh[h]), k64, True), (to_u16(vh[h]), v64, False)):
        ok = bf16_ulp_close(got, ref)
        if not ok.all():  # cancellation slack: 2^-20 x the summed magnitudes of the decoded terms
            a = (got.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
            slack = 2.0 ** -20 * decode_term_magnitude(ch, key)
            ok |= np.abs(a - ref) <= slack
        assert ok.all()


def check_attention(run, heads, rows):
    lay, qs, out = run["layer"], run["qs"], run["out"]
    worst = 0.0
    for h in heads:
        ref = oracle.attend_rows(qs[-1][h], rows, [chunk_head(c, h) for c in lay.chunks], 1 / math.sqrt(D))
        got = out[h].cpu().numpy()[rows].astype(np.float64)
        err = np.abs(got - ref).max() / math.sqrt(np.mean(ref ** 2))
        worst = max(worst, err)
        assert err <= 2e-2, (h, err)
    return worst
