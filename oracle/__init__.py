"""CPU oracle of the QuantWM quantise-and-attend path (ctypes front end of qwm_oracle.c).

TEST INFRASTRUCTURE ONLY.  Only `tests/`, `__graft_entry__.smoke()` and the
CPU-baseline leg of `bench.py` may import this package.  It shares nothing
with the CUDA library (`bit_kv_cache_qsac_gb300`) and never calls it.

Every function works on one head at a time and takes numpy arrays; bf16 and
fp16 values travel as their uint16 bit patterns.  The per-stage functions
follow the QuantWM summaries' step list ("方法步骤详情" steps 1-5 of the
Chinese summary; §4.1, §4.2, §C.3 and §D.1 of the v2 summary) and the QVG
summary's k-means smoothing (§2A) and warm start (§2C).

Parity pins: every function here is pinned by `tests/test_oracle_pins.py`
against closed forms, special cases, library routines or worked examples;
none is "parity unpinned".
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qwm_oracle.c")
_LIB_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_LIB_DIR, "liboracle.so")
_CFLAGS = ["-std=c11", "-O2", "-fopenmp", "-frounding-math", "-ffp-contract=off",
           "-fno-fast-math", "-shared", "-fPIC"]

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile qwm_oracle.c with gcc into oracle/_build/liboracle.so."""
    os.makedirs(_LIB_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *_CFLAGS, "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB)
    return _LIB


P = C.c_void_p
I64 = C.c_int64
I32 = C.c_int32


class QuantArgs(C.Structure):
    _fields_ = [
        ("k", P), ("v", P), ("cent_k", P), ("cent_v", P), ("w", P), ("M_full", P), ("u_r", P), ("u_r_f64", P),
        ("force_idx_k", P), ("force_idx_v", P),
        ("n", I64), ("d", I32), ("C", I32), ("group", I32), ("top_m", I32), ("rank", I32),
        ("storage", I32), ("psac_gate", I32),
        ("idx_k", P), ("idx_v", P), ("k_codes", P), ("v_codes", P),
        ("k_scale", P), ("k_min", P), ("v_scale", P), ("v_min", P),
        ("c", P), ("c_scale", P), ("c_real", P), ("cand", P), ("score2", P), ("dq_edge", P),
        ("vdist2", P), ("k_s8", P), ("v_s8", P), ("k_zp", P), ("v_zp", P), ("k_sigma", P), ("v_sigma", P),
        ("gate_err", P),
    ]


class ChunkHead(C.Structure):
    _fields_ = [
        ("n", I64), ("rank", I32),
        ("idx_k", P), ("idx_v", P), ("k_codes", P), ("v_codes", P),
        ("k_scale", P), ("k_min", P), ("v_scale", P), ("v_min", P),
        ("cent_k", P), ("cent_v", P), ("c", P), ("c_scale", P), ("u_r", P),
        ("k_raw", P), ("v_raw", P), ("causal_tpf", I64), ("cent_fp16", I32),
    ]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            l = C.CDLL(build())
            l.oracle_stats_accumulate.argtypes = [P, I64, C.c_int, P]
            l.oracle_weights.argtypes = [P, I64, C.c_int, P]
            l.oracle_eig_sym.argtypes = [P, C.c_int, C.c_double, C.c_int, P, P]
            l.oracle_eig_sym.restype = C.c_int
            l.oracle_basis_bf16.argtypes = [P, C.c_int, C.c_int, P]
            l.oracle_kmeans.argtypes = [P, I64, C.c_int, C.c_int, P, C.c_int, P, P, P, P]
            l.oracle_kmeans_objective.argtypes = [P, I64, C.c_int, P, C.c_int]
            l.oracle_kmeans_objective.restype = C.c_double
            l.oracle_int2_encode_group.argtypes = [P, C.c_int, P, P, P]
            l.oracle_pack2.argtypes = [P, C.c_int, P]
            l.oracle_int8_encode_token.argtypes = [P, C.c_int, P, P]
            l.oracle_quantize_head.argtypes = [C.POINTER(QuantArgs)]
            l.oracle_attend_rows.argtypes = [P, C.c_int, C.c_int, P, I64, C.POINTER(ChunkHead),
                                             C.c_int, C.c_double, P, P]
            l.oracle_dequantize_head.argtypes = [C.POINTER(ChunkHead), C.c_int, C.c_int, P, P, P, P]
            l.oracle_prq_residual.argtypes = [P, I64, C.c_int, P, P, P]
            l.oracle_kivi_quantize_head.argtypes = [P, P, I64, C.c_int, C.c_int, P, P, P, P, P, P]
            l.oracle_kivi_dequantize_head.argtypes = [P, P, P, P, P, P, I64, C.c_int, C.c_int, P, P]
            l.oracle_fp16_val.argtypes = [C.c_uint16]
            l.oracle_fp16_val.restype = C.c_double
            l.oracle_round_fp16.argtypes = [C.c_double, C.c_int]
            l.oracle_round_fp16.restype = C.c_double
            l.oracle_fp16_bits.argtypes = [C.c_double]
            l.oracle_fp16_bits.restype = C.c_uint16
            l.oracle_bf16_rne.argtypes = [C.c_double]
            l.oracle_bf16_rne.restype = C.c_uint16
            _lib = l
    return _lib


def _c(a, dtype):
    """Contiguous array of the given dtype (a copy only when needed)."""
    return np.ascontiguousarray(a, dtype=dtype)


def _p(a):
    return None if a is None else a.ctypes.data_as(P)


# ---------------------------------------------------------------- step 1: statistics


def stats_accumulate(q_bf16: np.ndarray, S: np.ndarray) -> None:
    """S += sum_q q q^T for one head (q: uint16 [nq][d]; S: float64 [d][d], updated in place)."""
    q = _c(q_bf16, np.uint16)
    assert S.dtype == np.float64 and S.flags.c_contiguous
    lib().oracle_stats_accumulate(_p(q), q.shape[0], q.shape[1], _p(S))


def weights(S: np.ndarray, n: int) -> np.ndarray:
    """w_c = S_cc / n, or 1 at cold start (n == 0)."""
    S = _c(S, np.float64)
    w = np.empty(S.shape[0], np.float64)
    lib().oracle_weights(_p(S), int(n), S.shape[0], _p(w))
    return w


def eig(M: np.ndarray, tol_rel: float = 1e-14, max_sweeps: int = 60):
    """(lambda descending, U with U[:, k] the k-th eigenvector, sweeps or -1)."""
    M = _c(M, np.float64)
    d = M.shape[0]
    lam = np.empty(d, np.float64)
    U = np.empty((d, d), np.float64)
    sweeps = lib().oracle_eig_sym(_p(M), d, tol_rel, max_sweeps, _p(lam), _p(U))
    return lam, U, sweeps


def basis_bf16(U: np.ndarray, r: int) -> np.ndarray:
    """First r eigenvectors rounded to bf16: uint16 [d][r]."""
    U = _c(U, np.float64)
    d = U.shape[0]
    out = np.empty((d, r), np.uint16)
    if r:
        lib().oracle_basis_bf16(_p(U), d, r, _p(out))
    return out


def update_query_stats(q_bf16: np.ndarray, S: np.ndarray, n: np.ndarray, rank: int):
    """All heads: fold q [H][nq][d] into S [H][d][d] (float64, in place) and n [H] (in place);
    return (w [H][d], eigvals [H][d], U_r bf16 [H][d][rank], U float64 [H][d][d], sweeps [H])."""
    H, nq, d = q_bf16.shape
    w = np.empty((H, d)); lam = np.empty((H, d)); ur = np.empty((H, d, rank), np.uint16)
    U = np.empty((H, d, d)); sweeps = np.empty(H, np.int64)
    for h in range(H):
        stats_accumulate(q_bf16[h], S[h])
        n[h] += nq
        w[h] = weights(S[h], int(n[h]))
        if n[h] > 0:
            lam[h], U[h], sweeps[h] = eig(S[h] / float(n[h]))
        else:
            lam[h], U[h], sweeps[h] = 0.0, np.eye(d), 0
        ur[h] = basis_bf16(U[h], rank)
    return w, lam, ur, U, sweeps


# ---------------------------------------------------------------- step 2a: k-means


def kmeans(x_bf16: np.ndarray, n_centroids: int, init_bf16: np.ndarray | None, iters: int):
    """Lloyd k-means of one head: returns (cent bf16 [C][d], cent float64, last assignment, objective per iteration)."""
    x = _c(x_bf16, np.uint16)
    n, d = x.shape
    init = None if init_bf16 is None else _c(init_bf16, np.uint16)
    cent = np.empty((n_centroids, d), np.uint16)
    cent64 = np.empty((n_centroids, d), np.float64)
    asg = np.empty(max(n, 1), np.int32)
    obj = np.empty(max(iters, 1), np.float64)
    lib().oracle_kmeans(_p(x), n, d, n_centroids, _p(init), iters, _p(cent), _p(cent64), _p(asg), _p(obj))
    return cent, cent64, asg[:n], obj[:iters]


def kmeans_objective(x_bf16: np.ndarray, cent_bf16: np.ndarray) -> float:
    x = _c(x_bf16, np.uint16)
    cent = _c(cent_bf16, np.uint16)
    return lib().oracle_kmeans_objective(_p(x), x.shape[0], x.shape[1], _p(cent), cent.shape[0])


# ---------------------------------------------------------------- steps 2-4: quantiser


def int2_encode_group(r: np.ndarray):
    """(codes uint8 [g], s fp16 bits, m fp16 bits) for one group of float32 residuals."""
    r = _c(r, np.float32)
    codes = np.empty(r.size, np.uint8)
    s = C.c_uint16()
    m = C.c_uint16()
    lib().oracle_int2_encode_group(_p(r), r.size, _p(codes), C.byref(s), C.byref(m))
    return codes, s.value, m.value


def pack2(codes: np.ndarray) -> np.ndarray:
    codes = _c(codes, np.uint8)
    out = np.empty(codes.size // 4, np.uint8)
    lib().oracle_pack2(_p(codes), codes.size, _p(out))
    return out


def int8_encode_token(Cf: np.ndarray):
    """(c int8 [r], sC fp16 bits) for one token's float32 PSAC coefficients."""
    Cf = _c(Cf, np.float32)
    c = np.empty(Cf.size, np.int8)
    sc = C.c_uint16()
    lib().oracle_int8_encode_token(_p(Cf), Cf.size, _p(c), C.byref(sc))
    return c, sc.value


def quantize_head(k, v, cent_k, cent_v, w=None, u_r=None, *, group=64, top_m=4, rank=None,
                  u_r_f64=None, force_idx_k=None, force_idx_v=None, storage=0, psac_gate=0, M_full=None):
    """QSAC Key assignment, nearest-centroid Value assignment, INT2 residuals and PSAC for one head.

    k, v: uint16 [n][d]; cent_k, cent_v: uint16 [C][d]; w: float [d] or None (uniform);
    u_r: uint16 [d][r] or None (PSAC off).  storage 0: fp16 step and offset per (token, group);
    storage 1: the compact metadata (8-bit step, 2-bit zero-point, power-of-two second-level scale
    per 128-token tile).  psac_gate: keep C only where it lowers the w-weighted error.  M_full
    ([d][d], with w = diag(M_full)): rank the top-M candidates by the full quadratic form (English v2
    summary §C.4 ablation).
    Returns a dict of every output and diagnostic."""
    k = _c(k, np.uint16); v = _c(v, np.uint16)
    cent_k = _c(cent_k, np.uint16); cent_v = _c(cent_v, np.uint16)
    n, d = k.shape
    Cn = cent_k.shape[0]
    if rank is None:
        rank = 0 if (u_r is None and u_r_f64 is None) else (u_r if u_r is not None else u_r_f64).shape[1]
    G = d // group
    w64 = None if w is None else _c(w, np.float64)
    mf = None if M_full is None else _c(M_full, np.float64)
    ur = None if u_r is None else _c(u_r, np.uint16)
    ur64 = None if u_r_f64 is None else _c(u_r_f64, np.float64)
    fk = None if force_idx_k is None else _c(force_idx_k, np.int32)
    fv = None if force_idx_v is None else _c(force_idx_v, np.int32)
    o = dict(
        idx_k=np.empty(n, np.int32), idx_v=np.empty(n, np.int32),
        k_codes=np.empty((n, d // 4), np.uint8), v_codes=np.empty((n, d // 4), np.uint8),
        k_scale=np.empty((n, G), np.uint16), k_min=np.empty((n, G), np.uint16),
        v_scale=np.empty((n, G), np.uint16), v_min=np.empty((n, G), np.uint16),
        c=np.zeros((n, max(rank, 1)), np.int8), c_scale=np.zeros(n, np.uint16),
        c_real=np.zeros((n, max(rank, 1)), np.float64),
        cand=np.empty((n, top_m), np.int32), score2=np.empty((n, 2)), dq_edge=np.empty((n, 2)),
        vdist2=np.empty((n, 2)),
        k_s8=np.zeros((n, G), np.uint8), v_s8=np.zeros((n, G), np.uint8),
        k_zp=np.zeros(n, np.uint8), v_zp=np.zeros(n, np.uint8),
        k_sigma=np.zeros(((n + 127) // 128, G), np.uint16), v_sigma=np.zeros(((n + 127) // 128, G), np.uint16),
        gate_err=np.zeros((n, 2)),
    )
    a = QuantArgs(k=_p(k), v=_p(v), cent_k=_p(cent_k), cent_v=_p(cent_v), w=_p(w64), M_full=_p(mf), u_r=_p(ur),
                  u_r_f64=_p(ur64), force_idx_k=_p(fk), force_idx_v=_p(fv), n=n, d=d, C=Cn,
                  group=group, top_m=top_m, rank=rank, storage=storage, psac_gate=psac_gate,
                  **{key: _p(val) for key, val in o.items()})
    if n:
        lib().oracle_quantize_head(C.byref(a))
    o["c"] = o["c"][:, :rank]
    o["c_real"] = o["c_real"][:, :rank]
    o["rank"] = rank
    return o


# ---------------------------------------------------------------- step 5: attention, decoder


def _chunk_struct(ch: dict, keep: list) -> ChunkHead:
    """ch: per-head dict with idx_k, idx_v, k_codes, v_codes, k_scale, k_min, v_scale, v_min,
    the codebooks (cent_k, cent_v as bf16 bits, or the stored cent_k16, cent_v16 as fp16 bits, which
    then take precedence) and, when rank > 0, c, c_scale, u_r; or, for the chunk still being
    generated (kept in bf16), k_raw and v_raw ([n][d] bf16 bits) and optionally causal_tpf (tokens
    per frame of the block-causal mask, 0 = none)."""
    def arr(name, dtype):
        a = _c(ch[name], dtype)
        keep.append(a)
        return _p(a)
    if "k_raw" in ch:
        return ChunkHead(n=int(np.asarray(ch["k_raw"]).shape[0]), rank=0, k_raw=arr("k_raw", np.uint16),
                         v_raw=arr("v_raw", np.uint16), causal_tpf=int(ch.get("causal_tpf", 0)))
    rank = int(ch.get("rank", 0))
    f16 = "cent_k16" in ch
    return ChunkHead(
        n=int(np.asarray(ch["idx_k"]).shape[0]), rank=rank,
        idx_k=arr("idx_k", np.int32), idx_v=arr("idx_v", np.int32),
        k_codes=arr("k_codes", np.uint8), v_codes=arr("v_codes", np.uint8),
        k_scale=arr("k_scale", np.uint16), k_min=arr("k_min", np.uint16),
        v_scale=arr("v_scale", np.uint16), v_min=arr("v_min", np.uint16),
        cent_k=arr("cent_k16" if f16 else "cent_k", np.uint16), cent_v=arr("cent_v16" if f16 else "cent_v", np.uint16),
        c=arr("c", np.int8) if rank else None, c_scale=arr("c_scale", np.uint16) if rank else None,
        u_r=arr("u_r", np.uint16) if rank else None, cent_fp16=1 if f16 else 0,
    )


def attend_rows(q_bf16: np.ndarray, rows, chunks: list[dict], scale: float, group: int = 64,
                with_lse: bool = False):
    """Attention output (float64 [len(rows)][d]) of the listed query rows of one head over
    every token of every chunk in `chunks` (per-head chunk dicts); with_lse: also the rows'
    base-2 log-sum-exp of the logits, (output, lse)."""
    q = _c(q_bf16, np.uint16)
    rows = _c(np.asarray(rows), np.int64)
    d = q.shape[1]
    keep: list = []
    arr = (ChunkHead * max(1, len(chunks)))(*[_chunk_struct(ch, keep) for ch in chunks])
    out = np.empty((rows.size, d), np.float64)
    lse = np.empty(rows.size, np.float64) if with_lse else None
    lib().oracle_attend_rows(_p(q), d, group, _p(rows), rows.size, arr, len(chunks), float(scale), _p(out),
                             _p(lse) if with_lse else None)
    return (out, lse) if with_lse else out


def dequantize_head(ch: dict, d: int = 128, group: int = 64):
    """(K_hat bf16 [n][d], V_hat bf16 [n][d], K_hat float64, V_hat float64) of one head of one chunk."""
    keep: list = []
    s = _chunk_struct(ch, keep)
    n = s.n
    kh = np.empty((n, d), np.uint16); vh = np.empty((n, d), np.uint16)
    kh64 = np.empty((n, d)); vh64 = np.empty((n, d))
    lib().oracle_dequantize_head(C.byref(s), d, group, _p(kh), _p(vh), _p(kh64), _p(vh64))
    return kh, vh, kh64, vh64


def fp16_val(bits) -> np.ndarray:
    """fp16 bit patterns -> float64 values."""
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def round_fp16(x: float, direction: int) -> float:
    return lib().oracle_round_fp16(float(x), int(direction))


def bf16_rne(x: float) -> int:
    return lib().oracle_bf16_rne(float(x))


# ---------------------------------------------------------------- comparison baselines


def prq_residual(x_bf16: np.ndarray, cent_bf16: np.ndarray, idx: np.ndarray) -> np.ndarray:
    """QVG progressive residual quantisation (Quant VideoGen summary §2B): the residual the next
    stage quantises, bf16(x - mu_idx) for one head (x uint16 [n][d], cent uint16 [C][d])."""
    x = _c(x_bf16, np.uint16); cent = _c(cent_bf16, np.uint16); ix = _c(idx, np.int32)
    n, d = x.shape
    out = np.empty_like(x)
    if n:
        lib().oracle_prq_residual(_p(x), n, d, _p(cent), _p(ix), _p(out))
    return out


def prq_head(k, v, cents_k: list, cents_v: list, group: int = 64):
    """A QVG-style chunk for one head: len(cents) nearest-centroid stages (stage s quantises the
    previous stage's residual with codebook cents[s]), then INT2 of the last residual.  Returns the
    per-stage indices, the final stage's quantize_head output and the decoded K_hat, V_hat (double):
    the sum of every stage's centroid and the INT2 reconstruction."""
    rk, rv = _c(k, np.uint16), _c(v, np.uint16)
    idx_k, idx_v = [], []
    for s in range(len(cents_k) - 1):
        o = quantize_head(rk, rv, cents_k[s], cents_v[s], None, None, group=group, top_m=1, rank=0)
        idx_k.append(o["idx_k"]); idx_v.append(o["idx_v"])
        rk = prq_residual(rk, cents_k[s], o["idx_k"])
        rv = prq_residual(rv, cents_v[s], o["idx_v"])
    last = quantize_head(rk, rv, cents_k[-1], cents_v[-1], None, None, group=group, top_m=1, rank=0)
    idx_k.append(last["idx_k"]); idx_v.append(last["idx_v"])
    ch = dict(idx_k=last["idx_k"], idx_v=last["idx_v"], k_codes=last["k_codes"], v_codes=last["v_codes"],
              k_scale=last["k_scale"], k_min=last["k_min"], v_scale=last["v_scale"], v_min=last["v_min"],
              cent_k=_c(cents_k[-1], np.uint16), cent_v=_c(cents_v[-1], np.uint16), rank=0)
    _, _, kh, vh = dequantize_head(ch, group=group)
    bf = lambda a: (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    for s in range(len(cents_k) - 1):
        kh = kh + bf(_c(cents_k[s], np.uint16)[idx_k[s]])
        vh = vh + bf(_c(cents_v[s], np.uint16)[idx_v[s]])
    return dict(idx_k=idx_k, idx_v=idx_v, last=last, k_hat=kh, v_hat=vh)


def kivi_quantize_head(k, v, group: int = 32):
    """KIVI-style INT2 of one head: Keys per channel over groups of `group` tokens, Values per token
    over groups of `group` channels (k, v uint16 bf16 [n][d])."""
    k = _c(k, np.uint16); v = _c(v, np.uint16)
    n, d = k.shape
    ng = (n + group - 1) // group
    o = dict(k_codes=np.zeros((n, d // 4), np.uint8), k_scale=np.zeros((ng, d), np.uint16),
             k_min=np.zeros((ng, d), np.uint16), v_codes=np.zeros((n, d // 4), np.uint8),
             v_scale=np.zeros((n, d // group), np.uint16), v_min=np.zeros((n, d // group), np.uint16))
    if n:
        lib().oracle_kivi_quantize_head(_p(k), _p(v), n, d, group, _p(o["k_codes"]), _p(o["k_scale"]),
                                        _p(o["k_min"]), _p(o["v_codes"]), _p(o["v_scale"]), _p(o["v_min"]))
    return o


def kivi_dequantize_head(o: dict, group: int = 32):
    """(K_hat, V_hat) as doubles [n][d] from kivi_quantize_head's output."""
    n, d4 = o["k_codes"].shape
    d = 4 * d4
    kh = np.empty((n, d)); vh = np.empty((n, d))
    arrs = {key: _c(o[key], np.uint8 if key.endswith("codes") else np.uint16) for key in o}
    if n:
        lib().oracle_kivi_dequantize_head(_p(arrs["k_codes"]), _p(arrs["k_scale"]), _p(arrs["k_min"]),
                                          _p(arrs["v_codes"]), _p(arrs["v_scale"]), _p(arrs["v_min"]), n, d,
                                          group, _p(kh), _p(vh))
    return kh, vh


# ---------------------------------------------------------------- PSAC rank per head, coefficient layouts
#
# The Chinese summary's critique ("独立分析的弱点", weakness three) notes that how much of the Query
# energy the top directions hold differs by model and layer, so one global r is a compromise; the
# English v2 summary (§C.2) reports that a larger r still helps.  The rank per (chunk, head) below is
# the plainest rule that follows from the eigenvalues the statistics step already computes: the
# smallest r whose top-r eigenvalues hold a given share of tr M.  The packed coefficient layouts
# follow the English v2 summary §D.1 ("selects the smaller dense or sparse coefficient layout,
# including sparse-index storage"): a token whose stored correction is zero (sC = 0: the gate of
# step (4) dropped it, or its coefficients were all zero) needs no row in the sparse layout.


def adaptive_rank(lam, r_max: int, energy: float) -> int:
    """Smallest r in 0..r_max whose r largest eigenvalues hold at least `energy` of their sum
    (tr M, summed in descending order in double precision); r_max when no r <= r_max does; 0 when
    the sum is not positive (no Query seen)."""
    lam = np.sort(np.asarray(lam, np.float64))[::-1]
    tr = 0.0
    for x in lam:
        tr += float(x)
    if not tr > 0.0:
        return 0
    cum = 0.0
    for r in range(r_max + 1):
        if cum >= energy * tr:
            return r
        if r < lam.size:
            cum += float(lam[r])
    return r_max


SPARSE_TILE = 128  # tokens per bitmap tile of the sparse layout


def psac_sparse_encode(c: np.ndarray, c_scale: np.ndarray):
    """Sparse layout of one head's coefficients: c int8 [n][r], c_scale fp16 bits [n] ->
    (mask uint32 [tiles][4]: bit b of word w of tile t set when token 128 t + 32 w + b keeps a
    row; tile_rank int32 [tiles]: kept tokens before tile t; rows int8 [K][r] and scales uint16 [K]
    of the kept tokens in token order).  A token keeps its row when its scale is not zero."""
    c = np.asarray(c, np.int8)
    sc = np.asarray(c_scale, np.uint16)
    n = sc.size
    tiles = (n + SPARSE_TILE - 1) // SPARSE_TILE
    keep = sc != 0
    mask = np.zeros((tiles, 4), np.uint32)
    for i in np.nonzero(keep)[0]:
        t, b = divmod(int(i), SPARSE_TILE)
        mask[t, b // 32] |= np.uint32(1 << (b % 32))
    tile_rank = np.zeros(tiles, np.int32)
    total = 0
    for t in range(tiles):
        tile_rank[t] = total
        total += int(keep[t * SPARSE_TILE:(t + 1) * SPARSE_TILE].sum())
    return mask, tile_rank, c[keep].copy(), sc[keep].copy()


def psac_sparse_decode(mask, tile_rank, rows, scales, n: int, r: int):
    """Dense (c int8 [n][r], c_scale uint16 [n]) of a sparse layout: token i's row is found from the
    bitmap alone (its tile's kept count plus the set bits below it in its tile)."""
    c = np.zeros((n, r), np.int8)
    sc = np.zeros(n, np.uint16)
    for i in range(n):
        t, b = divmod(i, SPARSE_TILE)
        w, bit = divmod(b, 32)
        if not (int(mask[t, w]) >> bit) & 1:
            continue
        below = sum(bin(int(mask[t, x])).count("1") for x in range(w)) + bin(int(mask[t, w]) & ((1 << bit) - 1)).count("1")
        slot = int(tile_rank[t]) + below
        c[i] = rows[slot]
        sc[i] = scales[slot]
    return c, sc


def psac_layout_bytes(n: int, rank: int, kept: int) -> tuple[int, int]:
    """Bytes of one head's coefficients (int8 rows of `rank` bytes and an fp16 scale per stored row)
    in the dense layout (every token) and in the sparse layout (kept tokens, plus a 16-byte bitmap
    and a 4-byte kept count per 128-token tile).  A head of rank 0 stores nothing."""
    if rank == 0:
        return 0, 0
    tiles = (n + SPARSE_TILE - 1) // SPARSE_TILE
    return n * (rank + 2), kept * (rank + 2) + tiles * 20


def psac_plan(n: int, ranks, kept):
    """Per head: (sparse?, rows stored) choosing the smaller layout (dense on a tie)."""
    plan = []
    for r, k in zip(ranks, kept):
        dense, sparse = psac_layout_bytes(n, int(r), int(k))
        use_sparse = int(r) > 0 and sparse < dense
        plan.append((use_sparse, (int(k) if use_sparse else n) if int(r) > 0 else 0))
    return plan


def codebook_fp16(cent_bf16: np.ndarray) -> np.ndarray:
    """The stored codebook: the fp16 value (round to nearest even) of every bf16 centroid element,
    as fp16 bit patterns.  Exact for magnitudes in [2^-17, 65504] and for 0."""
    x = (np.asarray(cent_bf16, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    out = np.empty(x.size, np.uint16)
    flat = x.ravel()
    for i in range(flat.size):
        out[i] = lib().oracle_fp16_bits(lib().oracle_round_fp16(float(flat[i]), 0))
    return out.reshape(np.shape(cent_bf16))
