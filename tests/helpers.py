"""Conversions between the CUDA path's torch tensors and the oracle's numpy arrays (tests only)."""
import numpy as np


def to_u16(t) -> np.ndarray:
    """A 16-bit torch tensor (bf16 / fp16 / int16) -> numpy uint16 bit patterns."""
    import torch
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def from_u16(a: np.ndarray, dtype, device="cuda"):
    """numpy uint16 bit patterns -> torch tensor of a 16-bit dtype on the device."""
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint16).view(np.int16)).to(device).view(dtype)


def compact_as_fp16(s8, zp, sigma, n: int):
    """Compact INT2 metadata of one head (steps s8 [n][G], zero-points zp [n], second-level scales
    sigma fp16 bits [tiles][G]) re-expressed exactly as fp16 step and offset bits: s = sigma s8 and
    m = -z s are fp16 values (sigma is a power of two), and m + s q = s (q - z)."""
    G = s8.shape[1]
    sig = np.asarray(sigma, np.uint16).view(np.float16).astype(np.float64)[np.arange(n) // 128]
    z = np.stack([(zp >> (2 * g)) & 3 for g in range(G)], 1).astype(np.float64)
    s = sig * s8.astype(np.float64)
    m = -z * s
    assert np.all(s.astype(np.float16).astype(np.float64) == s) and np.all(m.astype(np.float16).astype(np.float64) == m)
    return s.astype(np.float16).view(np.uint16), m.astype(np.float16).view(np.uint16)


def chunk_head(chunk, h: int) -> dict:
    """Per-head numpy view of a packed chunk, in the oracle's chunk dict format (compact metadata
    re-expressed exactly as fp16 step and offset)."""
    r = chunk.rank_eff
    n = chunk.n_tokens
    if getattr(chunk, "compact", False):
        ks, km = compact_as_fp16(chunk.k_s8[h].cpu().numpy(), chunk.k_zp[h].cpu().numpy()[:n], to_u16(chunk.k_sigma[h]), n)
        vs, vm = compact_as_fp16(chunk.v_s8[h].cpu().numpy(), chunk.v_zp[h].cpu().numpy()[:n], to_u16(chunk.v_sigma[h]), n)
    else:
        ks, km = to_u16(chunk.k_scale[h]), to_u16(chunk.k_min[h])
        vs, vm = to_u16(chunk.v_scale[h]), to_u16(chunk.v_min[h])
    d = dict(
        idx_k=chunk.k_idx[h].cpu().numpy().astype(np.int32), idx_v=chunk.v_idx[h].cpu().numpy().astype(np.int32),
        k_codes=chunk.k_codes[h].cpu().numpy(), v_codes=chunk.v_codes[h].cpu().numpy(),
        k_scale=ks, k_min=km, v_scale=vs, v_min=vm,
        cent_k16=to_u16(chunk.cent_k16[h]), cent_v16=to_u16(chunk.cent_v16[h]), rank=r,
    )
    if r:
        c, sc = psac_dense_head(chunk, h)
        d.update(c=c, c_scale=sc, u_r=to_u16(chunk.u_r[h])[:, :r])
    return d


def psac_dense_head(chunk, h: int):
    """One head's PSAC coefficients (int8 [n][rank_eff], fp16 bits [n]) of a chunk in either layout:
    the dense arrays, or the per-head layout read back through the oracle's sparse decoder (a head's
    rank r_h <= rank_eff: its columns past r_h are zero)."""
    import oracle
    r, n = chunk.rank_eff, chunk.n_tokens
    if getattr(chunk, "c_layout", 0) == 0:
        return chunk.c[h].cpu().numpy()[:, :r], to_u16(chunk.c_scale[h])
    c_off, s_off, rh, sparse = chunk.plan[h]
    c = np.zeros((n, r), np.int8)
    sc = np.zeros(n, np.uint16)
    if rh == 0:
        return c, sc
    allc = chunk.c.cpu().numpy()
    alls = to_u16(chunk.c_scale)
    if not sparse:
        c[:, :rh] = allc[c_off:c_off + n * rh].reshape(n, rh)
        sc[:] = alls[s_off:s_off + n]
        return c, sc
    mask = chunk.c_mask[h].cpu().numpy().view(np.uint32)
    trank = chunk.c_tile_rank[h].cpu().numpy()
    kept = int(bin_count(mask))
    rows = allc[c_off:c_off + kept * rh].reshape(kept, rh)
    c2, sc2 = oracle.psac_sparse_decode(mask, trank, rows, alls[s_off:s_off + kept], n, rh)
    c[:, :rh] = c2
    return c, sc2


def bin_count(mask) -> int:
    return sum(bin(int(x)).count("1") for x in np.asarray(mask).ravel())


def bf16_ulp_close(a_bits: np.ndarray, b: np.ndarray, ulps: float = 1.0) -> np.ndarray:
    """|bf16(a) - b| <= ulps * one bf16 step at the larger magnitude (elementwise mask)."""
    a = (a_bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    m = np.maximum(np.abs(a), np.abs(b))
    step = np.where(m > 0, 2.0 ** (np.floor(np.log2(np.maximum(m, 1e-300))) - 7), 2.0 ** -133)
    return np.abs(a - b) <= ulps * step


def decode_term_magnitude(ch: dict, key: bool, group: int = 64) -> np.ndarray:
    """Sum of the magnitudes of the terms the decoder adds for every element ([n][d]):
    |mu| + |m| + |s q| (+ sum_k |c_hat_k U_r[c, k]| for Keys).  An fp32 evaluation of a sum that
    cancels carries an error of a few fp32 units of this, whatever the result's own size."""
    f16 = lambda b: np.asarray(b, np.uint16).view(np.float16).astype(np.float64)
    bf = lambda b: (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    pre = "k" if key else "v"
    idx, codes = ch["idx_" + pre], ch[pre + "_codes"]
    n, d = codes.shape[0], 4 * codes.shape[1]
    q = np.zeros((n, d))
    for c in range(d):
        q[:, c] = (codes[:, c // 4] >> (2 * (c % 4))) & 3
    g = np.arange(d) // group
    s, m = f16(ch[pre + "_scale"])[:, g], f16(ch[pre + "_min"])[:, g]
    mu = f16(ch["cent_" + pre + "16"]) if ("cent_" + pre + "16") in ch else bf(ch["cent_" + pre])
    t = np.abs(mu[idx]) + np.abs(m) + np.abs(s * q)
    if key and ch["rank"]:
        chat = f16(ch["c_scale"])[:, None] * ch["c"].astype(np.float64)
        t += np.abs(chat) @ np.abs(bf(ch["u_r"])).T
    return t
