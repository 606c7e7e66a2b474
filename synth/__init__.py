"""Seeded synthetic workloads shaped like video-world-model KV caches.

This module only draws inputs.  It holds none of the quantise-and-attend
arithmetic, so both the CPU oracle and the CUDA path may take their inputs
from here.

Recipe (QuantWM summaries, "Method" and "Experimental setup" sections, and the
QVG summary, "Semantic-Aware Smoothing"): cached Keys of a video model cluster
along the spatio-temporal token grid, a few channels carry outliers, and the
Query energy concentrates in a handful of principal directions (more than 60%
in the top 8).

* Keys (and, independently, Values), per head:
  256 latent cluster means ~ N(0, I_d); every token (t, y, x) of the latent
  grid takes the cluster picked by a smooth random field (i.i.d. N(0, 1) on the
  grid, blurred by a periodic separable Gaussian with sigma_t = 1 frame and
  sigma_y = sigma_x = 2 tokens, then ranked so that each cluster owns an equal
  share of the grid), plus noise N(0, 0.3^2); eight channels chosen by a
  seeded permutation are multiplied by 8 after the noise is added.
* Queries, per head: q = A_h z + 0.3 eps with z ~ N(0, I_8) and
  A_h = alpha * G, G ~ N(0, 1)^{d x 8}, alpha chosen so that ||A_h||_F^2 = 19.34.
  Then E[q q^T] = A A^T + 0.09 I and the top-8 eigen-directions hold
  (19.34 + 8 * 0.09) / (19.34 + 128 * 0.09) = 0.65 of the energy.
  A_h is fixed per head; z and eps are fresh for every chunk of Queries.

Every array is returned as bfloat16 bit patterns (uint16, round to nearest
even), laid out [head][token][channel].

Seeds: each (config, layer, kind, head[, chunk]) tuple seeds its own PCG64
stream through numpy's SeedSequence, so any head or chunk can be drawn alone
and the draws do not depend on the order in which they are made.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

KIND_KEYS, KIND_VALUES, KIND_QMIX, KIND_QCHUNK = 0, 1, 2, 3

QUERY_SIGNAL_ENERGY = 19.34      # ||A_h||_F^2
QUERY_NOISE_STD = 0.3
KEY_NOISE_STD = 0.3
N_LATENT_CLUSTERS = 256
N_OUTLIER_CHANNELS = 8
OUTLIER_SCALE = 8.0
QUERY_RANK = 8


@dataclass(frozen=True)
class Workload:
    """Shape of one synthetic workload (one layer unless `layers` > 1)."""
    name: str
    config_id: int
    heads: int
    frames: int            # latent frames in the whole cache
    hs: int                # latent grid height (tokens)
    ws: int                # latent grid width (tokens)
    frames_per_chunk: int  # latent frames quantised per chunk
    nq_stats: int          # Queries folded into the statistics per step
    nq_attend: int         # Queries attending per step
    head_dim: int = 128
    n_centroids: int = 256
    group: int = 64
    top_m: int = 4
    rank: int = 8
    layers: int = 1
    extra: dict = field(default_factory=dict, compare=False, hash=False)

    @property
    def tokens_per_frame(self) -> int:
        return self.hs * self.ws

    @property
    def n_tokens(self) -> int:
        return self.frames * self.tokens_per_frame

    @property
    def chunk_tokens(self) -> int:
        return self.frames_per_chunk * self.tokens_per_frame

    @property
    def n_chunks(self) -> int:
        return self.frames // self.frames_per_chunk


# The five workloads.  "tiny" is one quantise step over 4 frames of 16x16;
# the 480p and 720p layers stream 8 chunks of 3 latent frames each.
TINY = Workload("tiny", 0, heads=2, frames=4, hs=16, ws=16, frames_per_chunk=4,
                nq_stats=256, nq_attend=256)
P480 = Workload("480p", 1, heads=40, frames=24, hs=30, ws=52, frames_per_chunk=3,
                nq_stats=4680, nq_attend=4680)
P720 = Workload("720p", 2, heads=40, frames=24, hs=45, ws=80, frames_per_chunk=3,
                nq_stats=10800, nq_attend=10800)
FULL_MODEL = Workload("480p-40-layers", 3, heads=40, frames=24, hs=30, ws=52,
                      frames_per_chunk=3, nq_stats=4680, nq_attend=4680, layers=40)
ABLATION = Workload("480p-ablation", 4, heads=40, frames=24, hs=30, ws=52,
                    frames_per_chunk=3, nq_stats=4680, nq_attend=4680)
WORKLOADS = {w.config_id: w for w in (TINY, P480, P720, FULL_MODEL, ABLATION)}


def _rng(*key: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(k) for k in key])))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even); return the bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bfloat16 bit patterns to float32 (exact)."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _periodic_gaussian_blur(field_: np.ndarray, sigmas) -> np.ndarray:
    """Separable periodic Gaussian blur, applied through the FFT of each axis."""
    out = np.fft.fftn(field_)
    for axis, sigma in enumerate(sigmas):
        n = field_.shape[axis]
        f = np.fft.fftfreq(n)
        kern = np.exp(-2.0 * (np.pi * sigma * f) ** 2)   # Fourier transform of a unit-mass Gaussian
        shape = [1] * field_.ndim
        shape[axis] = n
        out = out * kern.reshape(shape)
    return np.fft.ifftn(out).real


def cluster_ids(w: Workload, layer: int, kind: int, head: int) -> np.ndarray:
    """Latent cluster id of every token of the cache, in raster order (t, y, x)."""
    g = _rng(w.config_id, layer, kind, head, 0)
    noise = g.standard_normal((w.frames, w.hs, w.ws))
    smooth = _periodic_gaussian_blur(noise, (1.0, 2.0, 2.0)).reshape(-1)
    order = np.argsort(smooth, kind="stable")          # ties broken by linear index
    rank = np.empty_like(order)
    rank[order] = np.arange(order.size)
    return (N_LATENT_CLUSTERS * rank) // order.size


def _kv_head(w: Workload, layer: int, kind: int, head: int, t0: int, t1: int) -> np.ndarray:
    d = w.head_dim
    g_means = _rng(w.config_id, layer, kind, head, 1)
    means = g_means.standard_normal((N_LATENT_CLUSTERS, d), dtype=np.float32)
    outliers = g_means.permutation(d)[:N_OUTLIER_CHANNELS]
    ids = cluster_ids(w, layer, kind, head)[t0:t1]
    # noise for token j of the head comes from a stream keyed by the token's frame,
    # so a chunk can be drawn without drawing the frames before it
    fpt = w.tokens_per_frame
    out = np.empty((t1 - t0, d), dtype=np.float32)
    f0, f1 = t0 // fpt, (t1 + fpt - 1) // fpt
    for f in range(f0, f1):
        a, b = max(t0, f * fpt), min(t1, (f + 1) * fpt)
        eps = _rng(w.config_id, layer, kind, head, 2, f).standard_normal((fpt, d), dtype=np.float32)
        out[a - t0:b - t0] = eps[a - f * fpt:b - f * fpt]
    out *= np.float32(KEY_NOISE_STD)
    out += means[ids]
    out[:, outliers] *= np.float32(OUTLIER_SCALE)
    return f32_to_bf16_bits(out)


def _parallel_heads(fn, heads: int):
    workers = min(heads, max(1, (os.cpu_count() or 1)))
    with ThreadPoolExecutor(max_workers=workers) as ex:
        return list(ex.map(fn, range(heads)))


def keys(w: Workload, layer: int = 0, t0: int = 0, t1: int | None = None) -> np.ndarray:
    """Keys of tokens [t0, t1) of every head: uint16 (bf16) [H][t1 - t0][d]."""
    t1 = w.n_tokens if t1 is None else t1
    return np.stack(_parallel_heads(lambda h: _kv_head(w, layer, KIND_KEYS, h, t0, t1), w.heads))


def values(w: Workload, layer: int = 0, t0: int = 0, t1: int | None = None) -> np.ndarray:
    """Values of tokens [t0, t1) of every head: uint16 (bf16) [H][t1 - t0][d]."""
    t1 = w.n_tokens if t1 is None else t1
    return np.stack(_parallel_heads(lambda h: _kv_head(w, layer, KIND_VALUES, h, t0, t1), w.heads))


def query_mixing(w: Workload, layer: int, head: int) -> np.ndarray:
    """A_h in R^{d x 8}, scaled to ||A_h||_F^2 = 19.34."""
    g = _rng(w.config_id, layer, KIND_QMIX, head)
    G = g.standard_normal((w.head_dim, QUERY_RANK))
    return G * np.sqrt(QUERY_SIGNAL_ENERGY / np.sum(G * G))


def _q_head(w: Workload, layer: int, head: int, chunk: int, nq: int) -> np.ndarray:
    A = query_mixing(w, layer, head)
    g = _rng(w.config_id, layer, KIND_QCHUNK, head, chunk)
    z = g.standard_normal((nq, QUERY_RANK))
    eps = g.standard_normal((nq, w.head_dim))
    return f32_to_bf16_bits((z @ A.T + QUERY_NOISE_STD * eps).astype(np.float32))


def queries(w: Workload, chunk: int, nq: int, layer: int = 0) -> np.ndarray:
    """Fresh Queries of one chunk (chunk index >= 0): uint16 (bf16) [H][nq][d].

    By convention chunk index -1 is the calibration batch that precedes the
    tiny workload's single quantise step."""
    return np.stack(_parallel_heads(lambda h: _q_head(w, layer, h, chunk + 1, nq), w.heads))


def chunk_range(w: Workload, chunk: int) -> tuple[int, int]:
    """Token range [t0, t1) of a chunk (0-based) inside the cache."""
    n = w.chunk_tokens
    return chunk * n, (chunk + 1) * n


def unit_residuals(n: int, d: int, seed: int) -> np.ndarray:
    """Uniform(-1, 1) float32 residual rows, for quantiser error statistics."""
    return _rng(9999, seed).uniform(-1.0, 1.0, size=(n, d)).astype(np.float32)


def small_case(heads: int, n: int, d: int, n_centroids: int, nq: int, seed: int):
    """A small random case with the same distributions (for tests that sweep shapes):
    returns (k, v, q_stats, q_attend) as bf16 bit arrays."""
    frames = max(1, -(-n // 64))
    hs, ws = 8, 8
    w = Workload(f"small-{seed}", 100 + seed, heads=heads, frames=frames, hs=hs, ws=ws,
                 frames_per_chunk=frames, nq_stats=nq, nq_attend=nq, head_dim=d,
                 n_centroids=n_centroids)
    k = keys(w)[:, :n]
    v = values(w)[:, :n]
    return k, v, queries(w, -1, nq), queries(w, 0, nq)
