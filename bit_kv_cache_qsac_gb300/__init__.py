"""Python binding of libqwm.so, the GB300 (sm_103a) QuantWM quantise-and-attend library.

The functions mirror the C ABI in include/qwm.h one to one (same names, same
argument order) and only marshal arguments: every step of the path runs in the
library's CUDA kernels.  Tensors are torch CUDA tensors (PyTorch provides the
device memory and the stream); bf16 data may be torch.bfloat16 or 16-bit integer
tensors holding the bit patterns, fp16 data torch.float16 or 16-bit integers.

Importing this package loads the in-tree libqwm.so and raises when it is missing:
there is no fallback path.  Build it with `python -m bit_kv_cache_qsac_gb300.build`
(or `__graft_entry__.build()`).
"""
from __future__ import annotations

import ctypes as C
import os
from dataclasses import dataclass

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libqwm.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"libqwm.so not found at {LIB_PATH}: build it with "
                      "`python -m bit_kv_cache_qsac_gb300.build` before importing this package")

_lib = C.CDLL(LIB_PATH)

QWM_OK, QWM_ERR_ARG, QWM_ERR_SHAPE, QWM_ERR_ALIGN, QWM_ERR_CUDA, QWM_ERR_NOT_CONVERGED, \
    QWM_ERR_UNSUPPORTED, QWM_ERR_RANGE, QWM_ERR_DEVICE_TIMEOUT = range(9)

EXPORTED = ("qwm_status_string", "qwm_workspace_bytes", "qwm_create", "qwm_destroy",
            "qwm_update_query_stats", "qwm_fit_centroids", "qwm_fit_centroids_kv", "qwm_quantize_kv", "qwm_attend", "qwm_attend_merge",
            "qwm_dequantize", "qwm_sync_status", "qwm_update_query_stats_noalloc", "qwm_quantize_kv_full",
            "qwm_dequantize_chunks", "qwm_select_rank", "qwm_psac_kept", "qwm_psac_plan", "qwm_psac_pack",
            # comparison baselines (include/qwm_baselines.h)
            "qwm_kivi_quantize", "qwm_kivi_dequantize", "qwm_prq_residual", "qwm_prq_dequantize")


class QwmError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = _lib.qwm_status_string(status).decode()
        super().__init__(f"{where}: {msg} (status {status})")


class qwm_config(C.Structure):
    _fields_ = [("heads", C.c_int32), ("head_dim", C.c_int32), ("n_centroids", C.c_int32),
                ("group", C.c_int32), ("top_m", C.c_int32), ("rank", C.c_int32), ("bits", C.c_int32),
                ("kmeans_iters", C.c_int32), ("seed", C.c_uint64), ("storage", C.c_int32),
                ("psac_gate", C.c_int32), ("test_flags", C.c_int32)]


QWM_STORAGE_FP16, QWM_STORAGE_COMPACT = 0, 1
QWM_TEST_EXPIRE_WAIT = 1  # qwm_config.test_flags: one wait of qwm_attend runs out (tests of the error path)


class qwm_chunk(C.Structure):
    _fields_ = [("n_tokens", C.c_int64), ("rank_eff", C.c_int32), ("kind", C.c_int32),
                ("k_codes", C.c_void_p), ("v_codes", C.c_void_p), ("k_idx", C.c_void_p), ("v_idx", C.c_void_p),
                ("k_scale", C.c_void_p), ("k_min", C.c_void_p), ("v_scale", C.c_void_p), ("v_min", C.c_void_p),
                ("cent_k", C.c_void_p), ("cent_v", C.c_void_p), ("c", C.c_void_p), ("c_scale", C.c_void_p),
                ("u_r", C.c_void_p), ("cent_k16", C.c_void_p), ("cent_v16", C.c_void_p),
                ("k_raw", C.c_void_p), ("v_raw", C.c_void_p), ("causal_tpf", C.c_int64),
                ("k_s8", C.c_void_p), ("v_s8", C.c_void_p), ("k_zp", C.c_void_p), ("v_zp", C.c_void_p),
                ("k_sigma", C.c_void_p), ("v_sigma", C.c_void_p),
                ("c_layout", C.c_int32), ("c_heads", C.c_void_p), ("c_mask", C.c_void_p),
                ("c_tile_rank", C.c_void_p)]


QWM_C_DENSE, QWM_C_PER_HEAD = 0, 1


class qwm_psac_head(C.Structure):
    _fields_ = [("c_off", C.c_int64), ("s_off", C.c_int64), ("rank", C.c_int32), ("sparse", C.c_int32)]


QWM_CHUNK_PACKED, QWM_CHUNK_BF16 = 0, 1


class qwm_kivi_chunk(C.Structure):
    _fields_ = [("n_tokens", C.c_int64), ("k_codes", C.c_void_p), ("v_codes", C.c_void_p),
                ("k_scale", C.c_void_p), ("k_min", C.c_void_p), ("v_scale", C.c_void_p), ("v_min", C.c_void_p)]


class qwm_debug(C.Structure):
    _fields_ = [("c_f32", C.c_void_p), ("cand", C.c_void_p), ("score", C.c_void_p), ("gate_err", C.c_void_p)]


_P = C.c_void_p
_lib.qwm_status_string.argtypes = [C.c_int]
_lib.qwm_status_string.restype = C.c_char_p
_lib.qwm_workspace_bytes.argtypes = [C.POINTER(qwm_config)]
_lib.qwm_workspace_bytes.restype = C.c_size_t
_lib.qwm_create.argtypes = [C.POINTER(qwm_config), C.POINTER(C.c_void_p)]
_lib.qwm_destroy.argtypes = [_P]
_lib.qwm_update_query_stats.argtypes = [_P, _P, C.c_int64, _P, _P, _P, _P, _P, _P]
_lib.qwm_fit_centroids.argtypes = [_P, _P, C.c_int64, _P, _P, _P]
_lib.qwm_fit_centroids_kv.argtypes = [_P, _P, _P, C.c_int64, _P, _P, _P, _P, _P]
_lib.qwm_quantize_kv.argtypes = [_P, _P, _P, C.c_int64, _P, _P, C.POINTER(qwm_chunk), C.POINTER(qwm_debug), _P]
_lib.qwm_quantize_kv_full.argtypes = [_P, _P, _P, C.c_int64, _P, _P, _P, C.POINTER(qwm_chunk), C.POINTER(qwm_debug),
                                       _P]
_lib.qwm_attend.argtypes = [_P, _P, C.c_int64, C.POINTER(qwm_chunk), C.c_int32, C.c_float, _P, _P]
_lib.qwm_attend_merge.argtypes = [_P, _P, C.c_int64, C.POINTER(qwm_chunk), C.c_int32, C.c_float, _P, _P, C.c_int32, _P]
_lib.qwm_dequantize.argtypes = [_P, C.POINTER(qwm_chunk), _P, _P, _P]
_lib.qwm_dequantize_chunks.argtypes = [_P, C.POINTER(qwm_chunk), C.c_int32, _P, _P, _P]
_lib.qwm_select_rank.argtypes = [_P, _P, C.c_float, _P, _P, _P]
_lib.qwm_psac_kept.argtypes = [_P, C.POINTER(qwm_chunk), _P, _P]
_lib.qwm_psac_plan.argtypes = [C.POINTER(qwm_config), C.c_int64, _P, _P, C.POINTER(qwm_psac_head),
                               C.POINTER(C.c_int64), C.POINTER(C.c_int64)]
_lib.qwm_psac_pack.argtypes = [_P, C.POINTER(qwm_chunk), _P, _P, _P, _P, _P, _P]
_lib.qwm_sync_status.argtypes = [_P, _P]
_lib.qwm_update_query_stats_noalloc.argtypes = [C.POINTER(qwm_config), _P, C.c_int64, _P, _P, _P, _P, _P, _P, _P]
_lib.qwm_kivi_quantize.argtypes = [_P, _P, _P, C.c_int64, C.POINTER(qwm_kivi_chunk), _P]
_lib.qwm_kivi_dequantize.argtypes = [_P, C.POINTER(qwm_kivi_chunk), _P, _P, _P]
_lib.qwm_prq_residual.argtypes = [_P, _P, C.c_int64, _P, _P, _P, _P]
_lib.qwm_prq_dequantize.argtypes = [_P, C.POINTER(qwm_chunk), _P, _P, _P, _P, _P, _P, _P]
for _name in EXPORTED[2:]:
    getattr(_lib, _name).restype = C.c_int


def _check(status: int, where: str) -> None:
    if status != QWM_OK:
        raise QwmError(status, where)


def _stream(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


_WIDTH = {torch.bfloat16: 2, torch.float16: 2, torch.int16: 2, torch.uint16: 2, torch.float32: 4,
          torch.int32: 4, torch.int64: 8, torch.uint8: 1, torch.int8: 1}


def _ptr(t: torch.Tensor | None, name: str, width: int, shape: tuple | None = None) -> int | None:
    """Device pointer of a dense CUDA tensor with the given element width (and shape, when given)."""
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name}: expected a CUDA tensor")
    if _WIDTH.get(t.dtype) != width:
        raise TypeError(f"{name}: expected {width}-byte elements, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: tensor must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(t.shape)}")
    return t.data_ptr()


class Context:
    """Owns a qwm_ctx (its device workspace lives on the current device)."""

    def __init__(self, heads: int, n_centroids: int = 256, top_m: int = 4, rank: int = 8,
                 kmeans_iters: int = 10, head_dim: int = 128, group: int = 64, bits: int = 2,
                 storage: int = QWM_STORAGE_FP16, psac_gate: int = 0, test_flags: int = 0):
        self.cfg = qwm_config(heads, head_dim, n_centroids, group, top_m, rank, bits, kmeans_iters, 0, storage,
                              psac_gate, test_flags)
        h = C.c_void_p()
        _check(_lib.qwm_create(C.byref(self.cfg), C.byref(h)), "qwm_create")
        self.handle = h

    @property
    def heads(self):
        return self.cfg.heads

    def close(self):
        if self.handle:
            _check(_lib.qwm_destroy(self.handle), "qwm_destroy")
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def qwm_workspace_bytes(cfg: qwm_config) -> int:
    return _lib.qwm_workspace_bytes(C.byref(cfg))


@dataclass
class Chunk:
    """Device tensors of one packed chunk (all heads), mirroring qwm_chunk.  cent_k / cent_v are the
    bf16 codebooks the chunk is packed with (qwm_quantize_kv's input; `release_fit_codebooks` drops
    them); cent_k16 / cent_v16 are the chunk's stored codebooks."""
    n_tokens: int
    rank_eff: int
    k_codes: torch.Tensor
    v_codes: torch.Tensor
    k_idx: torch.Tensor
    v_idx: torch.Tensor
    k_scale: torch.Tensor
    k_min: torch.Tensor
    v_scale: torch.Tensor
    v_min: torch.Tensor
    cent_k: torch.Tensor | None
    cent_v: torch.Tensor | None
    c: torch.Tensor
    c_scale: torch.Tensor
    u_r: torch.Tensor
    cent_k16: torch.Tensor
    cent_v16: torch.Tensor
    # QWM_STORAGE_COMPACT contexts: 8-bit steps, 2-bit zero-points, per-tile second-level scales
    k_s8: torch.Tensor | None = None
    v_s8: torch.Tensor | None = None
    k_zp: torch.Tensor | None = None
    v_zp: torch.Tensor | None = None
    k_sigma: torch.Tensor | None = None
    v_sigma: torch.Tensor | None = None
    # per-head PSAC ranks (qwm_select_rank) and the per-head coefficient layout (qwm_psac_pack)
    head_rank: torch.Tensor | None = None    # int32 [H]
    c_layout: int = QWM_C_DENSE
    c_heads: torch.Tensor | None = None      # uint8 [H * 24]: the qwm_psac_head entries
    c_mask: torch.Tensor | None = None       # int32 (uint32 bits) [H][tiles][4]
    c_tile_rank: torch.Tensor | None = None  # int32 [H][tiles]
    plan: list | None = None                 # host copy of the entries: (c_off, s_off, rank, sparse)

    @property
    def compact(self) -> bool:
        return self.k_s8 is not None

    @staticmethod
    def empty(ctx: Context, n: int, device=None) -> "Chunk":
        cfg = ctx.cfg
        H, d, G, Cn, r = cfg.heads, cfg.head_dim, cfg.head_dim // cfg.group, cfg.n_centroids, cfg.rank
        dev = device or torch.device("cuda", torch.cuda.current_device())
        u8 = dict(dtype=torch.uint8, device=dev)
        f16 = dict(dtype=torch.float16, device=dev)
        ix = dict(dtype=torch.uint8 if Cn <= 256 else torch.int16, device=dev)  # int16 = uint16 bits
        books = (torch.empty(H, Cn, d, dtype=torch.bfloat16, device=dev),
                 torch.empty(H, Cn, d, dtype=torch.bfloat16, device=dev))
        psac = (torch.zeros(H, n, max(r, 1), dtype=torch.int8, device=dev), torch.zeros(H, n, **f16),
                torch.zeros(H, d, max(r, 1), dtype=torch.bfloat16, device=dev))
        stored = (torch.empty(H, Cn, d, **f16), torch.empty(H, Cn, d, **f16))
        if cfg.storage == QWM_STORAGE_COMPACT:
            nt = (n + 127) // 128
            z = lambda *shape, **kw: torch.zeros(*shape, **kw)
            return Chunk(n, 0,
                         torch.empty(H, n, d // 4, **u8), torch.empty(H, n, d // 4, **u8),
                         torch.empty(H, n, **ix), torch.empty(H, n, **ix),
                         z(0, **f16), z(0, **f16), z(0, **f16), z(0, **f16),
                         *books, *psac, *stored,
                         torch.empty(H, n, G, **u8), torch.empty(H, n, G, **u8),
                         torch.empty(H, max(n, 1), **u8), torch.empty(H, max(n, 1), **u8),
                         torch.empty(H, max(nt, 1), G, **f16), torch.empty(H, max(nt, 1), G, **f16))
        return Chunk(n, 0,
                     torch.empty(H, n, d // 4, **u8), torch.empty(H, n, d // 4, **u8),
                     torch.empty(H, n, **ix), torch.empty(H, n, **ix),
                     torch.empty(H, n, G, **f16), torch.empty(H, n, G, **f16),
                     torch.empty(H, n, G, **f16), torch.empty(H, n, G, **f16),
                     *books, *psac, *stored)

    def release_fit_codebooks(self) -> None:
        """Drop the bf16 codebooks (needed only by qwm_quantize_kv); the stored fp16 ones remain."""
        self.cent_k = None
        self.cent_v = None

    def nbytes(self) -> int:
        """Bytes of the packed representation: everything qwm_attend and qwm_dequantize read (codes,
        indices, INT2 metadata, stored codebooks, PSAC coefficients, their layout and the basis)."""
        meta = ((self.k_s8, self.v_s8, self.k_sigma, self.v_sigma) if self.compact
                else (self.k_scale, self.k_min, self.v_scale, self.v_min))
        nb = lambda ts: sum(t.numel() * t.element_size() for t in ts)
        tot = nb((self.k_codes, self.v_codes, self.k_idx, self.v_idx, self.cent_k16, self.cent_v16) + meta)
        if self.compact:  # the two groups' 2-bit zero-points of a token share one byte
            tot += self.k_zp.numel() + self.v_zp.numel()
        if self.rank_eff:
            tot += nb((self.c, self.c_scale, self.u_r))
            if self.c_layout == QWM_C_PER_HEAD:
                tot += nb((self.c_heads, self.c_mask, self.c_tile_rank))
        return tot

    def struct(self) -> qwm_chunk:
        def p(t, width):
            return _ptr(t, "chunk field", width)
        ph = self.c_layout == QWM_C_PER_HEAD
        return qwm_chunk(self.n_tokens, self.rank_eff, QWM_CHUNK_PACKED,
                         p(self.k_codes, 1), p(self.v_codes, 1),
                         p(self.k_idx, self.k_idx.element_size()), p(self.v_idx, self.v_idx.element_size()),
                         p(self.k_scale, 2), p(self.k_min, 2), p(self.v_scale, 2), p(self.v_min, 2),
                         p(self.cent_k, 2), p(self.cent_v, 2), p(self.c, 1), p(self.c_scale, 2), p(self.u_r, 2),
                         p(self.cent_k16, 2), p(self.cent_v16, 2),
                         None, None, 0,
                         *(p(t, w) for t, w in ((self.k_s8, 1), (self.v_s8, 1), (self.k_zp, 1), (self.v_zp, 1),
                                                (self.k_sigma, 2), (self.v_sigma, 2))),
                         self.c_layout, p(self.c_heads, 1) if ph else None, p(self.c_mask, 4) if ph else None,
                         p(self.c_tile_rank, 4) if ph else None)


@dataclass
class ActiveChunk:
    """The chunk still being generated: its bf16 Keys and Values [H][N][d], attended beside the
    packed chunks (qwm_chunk of kind QWM_CHUNK_BF16), with an optional block-causal mask over
    frames of `causal_tpf` tokens (Query row i is token i of this chunk)."""
    k: torch.Tensor
    v: torch.Tensor
    causal_tpf: int = 0

    @property
    def n_tokens(self) -> int:
        return self.k.shape[1]

    def struct(self) -> qwm_chunk:
        s = qwm_chunk()
        s.n_tokens, s.rank_eff, s.kind = self.n_tokens, 0, QWM_CHUNK_BF16
        s.k_raw = _ptr(self.k, "active chunk k", 2)
        s.v_raw = _ptr(self.v, "active chunk v", 2, tuple(self.k.shape))
        s.causal_tpf = int(self.causal_tpf)
        return s


def qwm_update_query_stats(ctx: Context, q, nq: int, S, n, w, eigvals, u_r, stream=None) -> None:
    H, d, r = ctx.cfg.heads, ctx.cfg.head_dim, ctx.cfg.rank
    st = _lib.qwm_update_query_stats(
        ctx.handle, _ptr(q, "q", 2, (H, nq, d)) if nq else None, nq,
        _ptr(S, "S", 4, (H, d, d)), _ptr(n, "n", 8, (H,)), _ptr(w, "w", 4, (H, d)),
        _ptr(eigvals, "eigvals", 4, (H, d)), _ptr(u_r, "u_r", 2, (H, d, r)) if r else None, _stream(stream))
    _check(st, "qwm_update_query_stats")


def qwm_fit_centroids(ctx: Context, x, n: int, init, cent, stream=None) -> None:
    H, d, Cn = ctx.cfg.heads, ctx.cfg.head_dim, ctx.cfg.n_centroids
    st = _lib.qwm_fit_centroids(ctx.handle, _ptr(x, "x", 2, (H, n, d)), n, _ptr(init, "init", 2, (H, Cn, d)),
                                _ptr(cent, "cent", 2, (H, Cn, d)), _stream(stream))
    _check(st, "qwm_fit_centroids")


def qwm_fit_centroids_kv(ctx: Context, k, v, n: int, init_k, init_v, cent_k, cent_v, stream=None) -> None:
    """The Key and Value codebooks of one chunk, the two fits side by side (same results as two
    qwm_fit_centroids calls)."""
    H, d, Cn = ctx.cfg.heads, ctx.cfg.head_dim, ctx.cfg.n_centroids
    st = _lib.qwm_fit_centroids_kv(ctx.handle, _ptr(k, "k", 2, (H, n, d)), _ptr(v, "v", 2, (H, n, d)), n,
                                   _ptr(init_k, "init_k", 2, (H, Cn, d)), _ptr(init_v, "init_v", 2, (H, Cn, d)),
                                   _ptr(cent_k, "cent_k", 2, (H, Cn, d)), _ptr(cent_v, "cent_v", 2, (H, Cn, d)),
                                   _stream(stream))
    _check(st, "qwm_fit_centroids_kv")


def qwm_quantize_kv(ctx: Context, k, v, n: int, w, u_r, out: Chunk, debug: dict | None = None,
                    stream=None) -> None:
    """Fill `out` (whose cent_k / cent_v hold the chunk's codebooks).  When u_r is given, out.u_r
    must be a tensor holding the same basis (the chunk keeps its own snapshot)."""
    H, d, r = ctx.cfg.heads, ctx.cfg.head_dim, ctx.cfg.rank
    s = out.struct()
    dbg = None
    if debug is not None:
        dbg = qwm_debug(_ptr(debug.get("c_f32"), "c_f32", 4), _ptr(debug.get("cand"), "cand", 4),
                        _ptr(debug.get("score"), "score", 4), _ptr(debug.get("gate_err"), "gate_err", 4))
    st = _lib.qwm_quantize_kv(ctx.handle, _ptr(k, "k", 2, (H, n, d)), _ptr(v, "v", 2, (H, n, d)), n,
                              _ptr(w, "w", 4, (H, d)), _ptr(u_r, "u_r", 2, (H, d, r)) if r else None,
                              C.byref(s), C.byref(dbg) if dbg is not None else None, _stream(stream))
    _check(st, "qwm_quantize_kv")
    out.rank_eff = s.rank_eff


def qwm_attend(ctx: Context, q, nq: int, chunks: list, softmax_scale: float, out, stream=None) -> None:
    H, d = ctx.cfg.heads, ctx.cfg.head_dim
    arr = (qwm_chunk * len(chunks))(*[c.struct() for c in chunks])
    st = _lib.qwm_attend(ctx.handle, _ptr(q, "q", 2, (H, nq, d)), nq, arr, len(chunks), float(softmax_scale),
                         _ptr(out, "out", 4, (H, nq, d)), _stream(stream))
    _check(st, "qwm_attend")


def qwm_attend_merge(ctx: Context, q, nq: int, chunks: list, softmax_scale: float, out, lse, merge: bool,
                     stream=None) -> None:
    """qwm_attend over some of a cache's chunks with the rows' log-sum-exp: merge=False writes out and
    lse; merge=True merges this call's chunks into the result already in out and lse."""
    H, d = ctx.cfg.heads, ctx.cfg.head_dim
    arr = (qwm_chunk * len(chunks))(*[c.struct() for c in chunks])
    st = _lib.qwm_attend_merge(ctx.handle, _ptr(q, "q", 2, (H, nq, d)), nq, arr, len(chunks), float(softmax_scale),
                               _ptr(out, "out", 4, (H, nq, d)), _ptr(lse, "lse", 4, (H, nq)), 1 if merge else 0,
                               _stream(stream))
    _check(st, "qwm_attend_merge")


def qwm_dequantize(ctx: Context, chunk: Chunk, k_hat, v_hat, stream=None) -> None:
    H, d = ctx.cfg.heads, ctx.cfg.head_dim
    s = chunk.struct()
    st = _lib.qwm_dequantize(ctx.handle, C.byref(s), _ptr(k_hat, "k_hat", 2, (H, chunk.n_tokens, d)),
                             _ptr(v_hat, "v_hat", 2, (H, chunk.n_tokens, d)), _stream(stream))
    _check(st, "qwm_dequantize")


def qwm_dequantize_chunks(ctx: Context, chunks, k_hat, v_hat, stream=None) -> None:
    """Decode several packed chunks in one launch into [H][sum N][d] (chunks in order)."""
    H, d = ctx.cfg.heads, ctx.cfg.head_dim
    total = sum(c.n_tokens for c in chunks)
    arr = (qwm_chunk * len(chunks))(*[c.struct() for c in chunks])
    st = _lib.qwm_dequantize_chunks(ctx.handle, arr, len(chunks), _ptr(k_hat, "k_hat", 2, (H, total, d)),
                                    _ptr(v_hat, "v_hat", 2, (H, total, d)), _stream(stream))
    _check(st, "qwm_dequantize_chunks")


def qwm_sync_status(ctx: Context, stream=None) -> int:
    """Wait for the stream and return (and clear) the first device-side error status (0 = none)."""
    return _lib.qwm_sync_status(ctx.handle, _stream(stream))


def qwm_update_query_stats_noalloc(cfg: qwm_config, q, nq: int, S, n, w, eigvals, u_r, dev_status=None,
                                   stream=None) -> None:
    """qwm_update_query_stats without a context and without any device allocation (for callers
    whose device memory is owned by someone else); see include/qwm.h."""
    H, d, r = cfg.heads, cfg.head_dim, cfg.rank
    st = _lib.qwm_update_query_stats_noalloc(
        C.byref(cfg), _ptr(q, "q", 2, (H, nq, d)) if nq else None, nq,
        _ptr(S, "S", 4, (H, d, d)), _ptr(n, "n", 8, (H,)), _ptr(w, "w", 4, (H, d)),
        _ptr(eigvals, "eigvals", 4, (H, d)), _ptr(u_r, "u_r", 2, (H, d, r)) if r else None,
        _ptr(dev_status, "dev_status", 4, (1,)), _stream(stream))
    _check(st, "qwm_update_query_stats_noalloc")


def qwm_select_rank(ctx: Context, eigvals, energy: float, u_r, head_rank, stream=None) -> None:
    """Per-head PSAC rank from the eigen-energy share (columns of u_r past each head's rank zeroed)."""
    H, d, r = ctx.cfg.heads, ctx.cfg.head_dim, ctx.cfg.rank
    st = _lib.qwm_select_rank(ctx.handle, _ptr(eigvals, "eigvals", 4, (H, d)), float(energy),
                              _ptr(u_r, "u_r", 2, (H, d, r)) if r else None, _ptr(head_rank, "head_rank", 4, (H,)),
                              _stream(stream))
    _check(st, "qwm_select_rank")


def qwm_psac_kept(ctx: Context, chunk: "Chunk", kept, stream=None) -> None:
    s = chunk.struct()
    st = _lib.qwm_psac_kept(ctx.handle, C.byref(s), _ptr(kept, "kept", 4, (ctx.cfg.heads,)), _stream(stream))
    _check(st, "qwm_psac_kept")


def qwm_psac_plan(cfg: qwm_config, n: int, head_rank, kept):
    """Host: (plan entries [(c_off, s_off, rank, sparse)] per head, bytes of c, scales of c_scale)."""
    H = cfg.heads
    hr = (C.c_int32 * H)(*[int(x) for x in head_rank])
    kp = (C.c_int32 * H)(*[int(x) for x in kept])
    plan = (qwm_psac_head * H)()
    cb, ns = C.c_int64(), C.c_int64()
    _check(_lib.qwm_psac_plan(C.byref(cfg), n, C.cast(hr, _P), C.cast(kp, _P), plan, C.byref(cb), C.byref(ns)),
           "qwm_psac_plan")
    return [(e.c_off, e.s_off, e.rank, e.sparse) for e in plan], cb.value, ns.value, bytes(plan)


def qwm_psac_pack(ctx: Context, dense: "Chunk", plan_dev, c, c_scale, c_mask, c_tile_rank, stream=None) -> None:
    s = dense.struct()
    st = _lib.qwm_psac_pack(ctx.handle, C.byref(s), _ptr(plan_dev, "plan", 1), _ptr(c, "c", 1),
                            _ptr(c_scale, "c_scale", 2), _ptr(c_mask, "c_mask", 4), _ptr(c_tile_rank, "c_tile_rank", 4),
                            _stream(stream))
    _check(st, "qwm_psac_pack")


def pack_psac_layout(ctx: Context, chunk: "Chunk", head_rank=None, stream=None) -> None:
    """Repack a dense chunk's PSAC coefficients into the per-head layout (each head its rank r_h and
    the smaller of the dense and sparse layouts): count the kept tokens per head, plan on the host
    (a synchronisation), allocate exactly the planned buffers, pack.  head_rank: device int32 [H]
    (qwm_select_rank's output), or None for config.rank on every head."""
    if not chunk.rank_eff or chunk.c_layout != QWM_C_DENSE or chunk.n_tokens == 0:
        return
    cfg = ctx.cfg
    H, n = cfg.heads, chunk.n_tokens
    dev = chunk.c.device
    kept = torch.empty(H, dtype=torch.int32, device=dev)
    qwm_psac_kept(ctx, chunk, kept, stream)
    (stream if stream is not None else torch.cuda.current_stream(dev)).synchronize()
    ranks = head_rank.cpu().tolist() if head_rank is not None else [chunk.rank_eff] * H
    plan, c_bytes, n_scales, raw = qwm_psac_plan(cfg, n, ranks, kept.cpu().tolist())
    tiles = (n + 127) // 128
    plan_dev = torch.frombuffer(bytearray(raw), dtype=torch.uint8).to(dev)
    c = torch.zeros(max(c_bytes, 1), dtype=torch.int8, device=dev)
    sc = torch.zeros(max(n_scales, 1), dtype=torch.float16, device=dev)
    mask = torch.zeros(H, tiles, 4, dtype=torch.int32, device=dev)
    trank = torch.zeros(H, tiles, dtype=torch.int32, device=dev)
    qwm_psac_pack(ctx, chunk, plan_dev, c, sc, mask, trank, stream)
    chunk.c, chunk.c_scale = c, sc
    chunk.c_heads, chunk.c_mask, chunk.c_tile_rank = plan_dev, mask, trank
    chunk.c_layout, chunk.plan = QWM_C_PER_HEAD, plan
    if head_rank is not None:
        chunk.head_rank = head_rank


def qwm_status_string(status: int) -> str:
    return _lib.qwm_status_string(status).decode()


def raw_library() -> C.CDLL:
    """The loaded libqwm.so (for tests that inspect its exported symbols)."""
    return _lib


# ---------------------------------------------------------------- comparison baselines (qwm_baselines.h)

KIVI_GROUP = 32


@dataclass
class KiviChunk:
    """Device tensors of one KIVI-style INT2 chunk (all heads), mirroring qwm_kivi_chunk."""
    n_tokens: int
    k_codes: torch.Tensor
    v_codes: torch.Tensor
    k_scale: torch.Tensor
    k_min: torch.Tensor
    v_scale: torch.Tensor
    v_min: torch.Tensor

    @staticmethod
    def empty(ctx: Context, n: int, device=None) -> "KiviChunk":
        H, d = ctx.cfg.heads, ctx.cfg.head_dim
        dev = device or torch.device("cuda", torch.cuda.current_device())
        ng = (n + KIVI_GROUP - 1) // KIVI_GROUP
        u8 = dict(dtype=torch.uint8, device=dev)
        f16 = dict(dtype=torch.float16, device=dev)
        return KiviChunk(n, torch.empty(H, n, d // 4, **u8), torch.empty(H, n, d // 4, **u8),
                         torch.empty(H, ng, d, **f16), torch.empty(H, ng, d, **f16),
                         torch.empty(H, n, d // KIVI_GROUP, **f16), torch.empty(H, n, d // KIVI_GROUP, **f16))

    def nbytes(self) -> int:
        return sum(t.numel() * t.element_size() for t in (self.k_codes, self.v_codes, self.k_scale, self.k_min,
                                                          self.v_scale, self.v_min))

    def struct(self) -> qwm_kivi_chunk:
        def p(t, width):
            return _ptr(t, "kivi chunk field", width)
        return qwm_kivi_chunk(self.n_tokens, p(self.k_codes, 1), p(self.v_codes, 1), p(self.k_scale, 2),
                              p(self.k_min, 2), p(self.v_scale, 2), p(self.v_min, 2))


def qwm_kivi_quantize(ctx: Context, k, v, n: int, out: KiviChunk, stream=None) -> None:
    H, d = ctx.cfg.heads, ctx.cfg.head_dim
    s = out.struct()
    _check(_lib.qwm_kivi_quantize(ctx.handle, _ptr(k, "k", 2, (H, n, d)), _ptr(v, "v", 2, (H, n, d)), n,
                                  C.byref(s), _stream(stream)), "qwm_kivi_quantize")


def qwm_kivi_dequantize(ctx: Context, chunk: KiviChunk, k_hat, v_hat, stream=None) -> None:
    H, d = ctx.cfg.heads, ctx.cfg.head_dim
    s = chunk.struct()
    _check(_lib.qwm_kivi_dequantize(ctx.handle, C.byref(s), _ptr(k_hat, "k_hat", 2, (H, chunk.n_tokens, d)),
                                    _ptr(v_hat, "v_hat", 2, (H, chunk.n_tokens, d)), _stream(stream)),
           "qwm_kivi_dequantize")


def qwm_prq_residual(ctx: Context, x, n: int, cent, idx, out, stream=None) -> None:
    H, d, Cn = ctx.cfg.heads, ctx.cfg.head_dim, ctx.cfg.n_centroids
    _check(_lib.qwm_prq_residual(ctx.handle, _ptr(x, "x", 2, (H, n, d)), n, _ptr(cent, "cent", 2, (H, Cn, d)),
                                 _ptr(idx, "idx", idx.element_size(), (H, n)), _ptr(out, "out", 2, (H, n, d)),
                                 _stream(stream)), "qwm_prq_residual")


def qwm_prq_dequantize(ctx: Context, last: Chunk, cent1_k, idx1_k, cent1_v, idx1_v, k_hat, v_hat,
                       stream=None) -> None:
    H, d, Cn, n = ctx.cfg.heads, ctx.cfg.head_dim, ctx.cfg.n_centroids, last.n_tokens
    s = last.struct()
    _check(_lib.qwm_prq_dequantize(ctx.handle, C.byref(s), _ptr(cent1_k, "cent1_k", 2, (H, Cn, d)),
                                   _ptr(idx1_k, "idx1_k", idx1_k.element_size(), (H, n)),
                                   _ptr(cent1_v, "cent1_v", 2, (H, Cn, d)),
                                   _ptr(idx1_v, "idx1_v", idx1_v.element_size(), (H, n)),
                                   _ptr(k_hat, "k_hat", 2, (H, n, d)), _ptr(v_hat, "v_hat", 2, (H, n, d)),
                                   _stream(stream)), "qwm_prq_dequantize")


def qwm_quantize_kv_full(ctx: Context, k, v, n: int, S, n_seen, u_r, out: Chunk, debug: dict | None = None,
                         stream=None) -> None:
    """qwm_quantize_kv with the QSAC candidates ranked by (k - mu)^T M (k - mu), M = S / n_seen formed
    by the library from the running statistics (S fp32 [H][d][d], n_seen int64 [H])."""
    H, d, r = ctx.cfg.heads, ctx.cfg.head_dim, ctx.cfg.rank
    s = out.struct()
    dbg = None
    if debug is not None:
        dbg = qwm_debug(_ptr(debug.get("c_f32"), "c_f32", 4), _ptr(debug.get("cand"), "cand", 4),
                        _ptr(debug.get("score"), "score", 4), _ptr(debug.get("gate_err"), "gate_err", 4))
    st = _lib.qwm_quantize_kv_full(ctx.handle, _ptr(k, "k", 2, (H, n, d)), _ptr(v, "v", 2, (H, n, d)), n,
                                   _ptr(S, "S", 4, (H, d, d)), _ptr(n_seen, "n_seen", 8, (H,)),
                                   _ptr(u_r, "u_r", 2, (H, d, r)) if r else None,
                                   C.byref(s), C.byref(dbg) if dbg is not None else None, _stream(stream))
    _check(st, "qwm_quantize_kv_full")
    out.rank_eff = s.rank_eff
