"""Chunk-streaming driver of one attention layer's compressed KV cache.

QuantWM processes the cache chunk by chunk (English v2 summary §5.1 and §D.1;
Chinese summary steps (1)-(5)): at each chunk boundary the previous chunk's
Queries are folded into the per-head statistics and the principal basis is
recomputed, the new chunk's Keys and Values are packed once, and the Queries of
the step attend over every packed chunk.  The first chunk has no statistics
(uniform weights, PSAC off).  This module only sequences the library calls; all
arithmetic runs in libqwm.so.
"""
from __future__ import annotations

import math

import torch

from . import (ActiveChunk, Chunk, Context, pack_psac_layout, qwm_attend, qwm_attend_merge, qwm_dequantize,
               qwm_fit_centroids_kv,
               qwm_quantize_kv, qwm_quantize_kv_full, qwm_select_rank, qwm_sync_status, qwm_update_query_stats)


class CompressedLayer:
    """Running state of one layer: Query statistics, basis, packed chunks, last codebooks."""

    def __init__(self, ctx: Context, device=None, full_query: bool = False, rank_energy: float | None = None,
                 psac_per_head: bool = False, keep_fit_codebooks: bool = False):
        """full_query: rank the QSAC candidates by the full Query second moment (English v2 §C.4
        ablation) instead of its diagonal.  rank_energy: choose each head's PSAC rank per chunk as the
        smallest r <= config.rank whose top-r eigenvalues hold this share of tr M (qwm_select_rank);
        implies the per-head coefficient layout.  psac_per_head: repack each chunk's coefficients into
        the per-head layout (the smaller of dense and sparse per head).  keep_fit_codebooks: keep
        every chunk's bf16 codebooks (only the packing reads them; by default only the last chunk's
        stay, as the next chunk's k-means start)."""
        self.ctx = ctx
        self.full_query = full_query
        self.rank_energy = rank_energy
        self.psac_per_head = psac_per_head or rank_energy is not None
        self.keep_fit_codebooks = keep_fit_codebooks
        cfg = ctx.cfg
        H, d, r = cfg.heads, cfg.head_dim, cfg.rank
        dev = device or torch.device("cuda", torch.cuda.current_device())
        self.device = dev
        self.S = torch.zeros(H, d, d, dtype=torch.float32, device=dev)
        self.n = torch.zeros(H, dtype=torch.int64, device=dev)
        self.w = torch.ones(H, d, dtype=torch.float32, device=dev)
        self.eigvals = torch.zeros(H, d, dtype=torch.float32, device=dev)
        self.u_r = torch.zeros(H, d, max(r, 1), dtype=torch.bfloat16, device=dev)
        self.n_seen = 0          # Queries folded in so far (host copy of n)
        self.chunks: list[Chunk] = []
        self.prev_cent_k = None
        self.prev_cent_v = None
        self._side = None        # second stream for the statistics update of step()
        self._stats_pending = None  # stream_step(): the fold the next packing waits for
        self._hist = None        # stream_step(overlap=True): high-priority stream of the history attention

    def fold_queries(self, q: torch.Tensor, stream=None) -> None:
        """Step 1: fold Queries [H][nq][d] into the statistics and recompute w and U_r."""
        nq = q.shape[1] if q is not None else 0
        qwm_update_query_stats(self.ctx, q, nq, self.S, self.n, self.w, self.eigvals,
                               self.u_r if self.ctx.cfg.rank else None, stream)
        self.n_seen += nq

    def append_chunk(self, k: torch.Tensor, v: torch.Tensor, warm_start: bool = True, stream=None,
                     debug: dict | None = None, stats_done=None) -> Chunk:
        """Steps 2-4: fit the chunk's codebooks and pack its Keys and Values.  `stats_done`: an
        event the packing waits for (a statistics update running on another stream)."""
        n = k.shape[1]
        ch = Chunk.empty(self.ctx, n, self.device)
        init_k = self.prev_cent_k if warm_start else None
        init_v = self.prev_cent_v if warm_start else None
        qwm_fit_centroids_kv(self.ctx, k, v, n, init_k, init_v, ch.cent_k, ch.cent_v, stream)
        s = stream if stream is not None else torch.cuda.current_stream(self.device)
        if stats_done is not None:
            s.wait_event(stats_done)
        psac = self.n_seen > 0 and self.ctx.cfg.rank > 0
        head_rank = None
        if psac:
            with torch.cuda.stream(s):
                ch.u_r.copy_(self.u_r)   # per-chunk snapshot of the basis
            if self.rank_energy is not None:   # per-head rank: basis columns past it zeroed
                head_rank = torch.empty(self.ctx.cfg.heads, dtype=torch.int32, device=self.device)
                qwm_select_rank(self.ctx, self.eigvals, self.rank_energy, ch.u_r, head_rank, stream)
        w = self.w if self.n_seen > 0 else None
        if self.full_query and w is not None:
            qwm_quantize_kv_full(self.ctx, k, v, n, self.S, self.n, ch.u_r if psac else None, ch, debug, stream)
        else:
            qwm_quantize_kv(self.ctx, k, v, n, w, ch.u_r if psac else None, ch, debug, stream)
        if psac and self.psac_per_head:
            pack_psac_layout(self.ctx, ch, head_rank, stream)
        self.chunks.append(ch)
        self.prev_cent_k, self.prev_cent_v = ch.cent_k, ch.cent_v
        if not self.keep_fit_codebooks:
            ch.release_fit_codebooks()   # the stored fp16 codebooks remain; prev_cent_* keeps this one
        return ch

    def attend(self, q: torch.Tensor, out: torch.Tensor | None = None, scale: float | None = None,
               stream=None, active: "ActiveChunk | None" = None) -> torch.Tensor:
        """Step 5: attention of Queries [H][nq][d] over every packed chunk and, when given, the
        chunk still being generated (bf16, optionally block-causal) in the same softmax."""
        H, nq, d = q.shape
        if out is None:
            out = torch.empty(H, nq, d, dtype=torch.float32, device=q.device)
        chunks = self.chunks + ([active] if active is not None else [])
        qwm_attend(self.ctx, q, nq, chunks, 1.0 / math.sqrt(d) if scale is None else scale, out, stream)
        return out

    def dequantize(self, i: int, stream=None):
        ch = self.chunks[i]
        H, d = self.ctx.cfg.heads, self.ctx.cfg.head_dim
        kh = torch.empty(H, ch.n_tokens, d, dtype=torch.bfloat16, device=self.device)
        vh = torch.empty_like(kh)
        qwm_dequantize(self.ctx, ch, kh, vh, stream)
        return kh, vh

    def step(self, q_prev, k, v, q, stream=None) -> torch.Tensor:
        """One streaming step: fold q_prev (may be None), pack (k, v), attend with q.

        The statistics update and the codebook fits do not depend on each other, so the statistics
        run on a second stream beside the fits; the packing waits for both."""
        main = stream if stream is not None else torch.cuda.current_stream(self.device)
        done = None
        if q_prev is not None:
            if self._side is None:
                self._side = torch.cuda.Stream(self.device)
            self._side.wait_stream(main)
            q_prev.record_stream(self._side)
            self.fold_queries(q_prev, self._side)
            done = torch.cuda.Event()
            done.record(self._side)
        self.append_chunk(k, v, stream=main, stats_done=done)
        return self.attend(q, stream=main)

    def stream_step(self, k, v, q, stream=None, overlap: bool = False) -> torch.Tensor:
        """One streaming step in pipelined order: pack (k, v) with the statistics of every Query
        folded so far, attend with q, and fold q into the statistics on a second stream while the
        attention runs; the next call's packing waits for that fold.  The same work as
        step(q_prev, k, v, q) with q_prev the previous call's q, with the statistics beside the
        attention instead of beside the codebook fits.

        overlap: the attention over the chunks already in the cache runs on a high-priority stream
        beside the new chunk's fits and packing (it does not depend on them), and the new chunk's
        attention then merges into it through the rows' log-sum-exp (qwm_attend_merge); the same
        output up to rounding."""
        main = stream if stream is not None else torch.cuda.current_stream(self.device)
        H, nq, d = q.shape
        scale = 1.0 / math.sqrt(d)
        history = None
        if overlap and self.chunks:
            if self._hist is None:
                self._hist = torch.cuda.Stream(self.device, priority=-1)
            out = torch.empty(H, nq, d, dtype=torch.float32, device=q.device)
            lse = torch.empty(H, nq, dtype=torch.float32, device=q.device)
            self._hist.wait_stream(main)
            for t in (q, out, lse):
                t.record_stream(self._hist)
            qwm_attend_merge(self.ctx, q, nq, list(self.chunks), scale, out, lse, False, self._hist)
            history = True
        self.append_chunk(k, v, stream=main, stats_done=self._stats_pending)
        packed = torch.cuda.Event()
        packed.record(main)
        if self._side is None:
            self._side = torch.cuda.Stream(self.device)
        self._side.wait_event(packed)          # the packing has read w and the basis
        q.record_stream(self._side)
        self.fold_queries(q, self._side)
        self._stats_pending = torch.cuda.Event()
        self._stats_pending.record(self._side)
        if history is not None:
            # the new chunk merged in on the same high-priority stream (the statistics fold beside it
            # fills the SMs it leaves)
            self._hist.wait_event(packed)
            qwm_attend_merge(self.ctx, q, nq, [self.chunks[-1]], scale, out, lse, True, self._hist)
            main.wait_stream(self._hist)
        else:
            out = self.attend(q, stream=main)
        main.wait_event(self._stats_pending)   # the step ends when both are done
        return out

    def check(self, stream=None) -> int:
        return qwm_sync_status(self.ctx, stream)

    def nbytes(self) -> int:
        return sum(c.nbytes() for c in self.chunks)
