"""Plain, slow reference of every step of the indexer hot path (numpy, f64).

Test infrastructure only (see the package docstring). bf16 tensors are
carried as numpy uint16 bit patterns; all arithmetic is f64 unless a step's
precision is fixed (the RoPE rotation is f32, see rope_interleaved).
"""
from __future__ import annotations

import math
from typing import Optional

import numpy as np

__all__ = [
    "FP4_BLOCK", "E2M1_GRID", "KEY_ROW_BYTES", "SCALE_FLOOR", "key_row_bytes", "f32_to_bf16",
    "bf16_to_f64", "f64_to_bf16", "yarn_freqs_cis", "linear_bf16", "rmsnorm_bf16",
    "rope_interleaved", "fp4_quant_e8m0", "pack_row68", "unpack_row68", "dequant_row68",
    "key_slots", "publish_keys", "project_queries", "prep_queries", "visible_lens", "index_scores",
    "select_candidate_blocks", "candidate_mask", "topk_positions", "forward",
    "FP8_BLOCK", "E4M3_GRID", "FP8_SCALE_FLOOR", "FP8_ROW_BYTES", "fp8_quant_ue8m0", "pack_row132",
    "dequant_row132", "dequant_row", "quantise_rows",
    "LATENT_BLOCK", "LATENT_SCALE_FLOOR", "e4m3_round", "fp4_quant_e4m3", "weights_proj", "compress_latent",
]

# fp4_block_size (compress module page, constant FP4_BLOCK).
FP4_BLOCK = 32
# The e2m1 magnitudes, indexed by the 3-bit magnitude code (OCP MX e2m1 format).
E2M1_GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
# amax floor of the e8m0 quantiser (compress module page, fp4_quant_e8m0_inplace).
SCALE_FLOOR = 6.0 * 2.0 ** -126


def key_row_bytes(head_dim: int) -> int:
    """68 for head_dim 128: packed nibbles + one UE8M0 byte per 32 values
    (attention.py patch page, _indexer_k_cache_head_dim, MXFP4 branch)."""
    return head_dim // 2 + head_dim // FP4_BLOCK


KEY_ROW_BYTES = key_row_bytes(128)


# ----------------------------------------------------------------------------- bf16
def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> exact f64 values."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def f64_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round f64 values to bf16 once, to nearest with ties to even (no f32 step).

    bf16 keeps 8 significant bits; below 2**-126 the quantum is fixed at 2**-133
    (subnormals). Results past the largest finite bf16 become infinities.
    """
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    _, e = np.frexp(a)                      # a = m * 2**e with m in [0.5, 1)
    quantum_exp = np.maximum(e, -125) - 8   # 8 significant bits
    r = np.ldexp(np.rint(np.ldexp(a, -quantum_exp)), quantum_exp)   # rint: ties to even
    r = np.where(a == 0, 0.0, r)
    big = r >= 2.0 ** 128
    r32 = np.where(big, np.inf, r).astype(np.float32)   # exact: r has <= 8 significant bits
    bits = (r32.view(np.uint32) >> 16).astype(np.uint16)
    sign = np.signbit(x).astype(np.uint16) << 15
    return bits | sign


def f32_to_bf16(x32: np.ndarray) -> np.ndarray:
    return f64_to_bf16(np.asarray(x32, dtype=np.float32).astype(np.float64))


# ----------------------------------------------------------------------------- YaRN
def yarn_freqs_cis(rope_dim: int, max_pos: int, theta: float, factor: float, original_seq_len: int,
                   beta_fast: float, beta_slow: float):
    """cos / sin tables [max_pos][rope_dim/2] (f32) of the YaRN RoPE.

    compress module page, yarn_freqs_cis: precompute_freqs_cis WITH YaRN when
    original_seq_len > 0, built from compress_rope_theta, result [seqlen][dim/2]
    of (cos, sin). The body is not on the pages; this follows the published
    YaRN "NTK-by-parts" interpolation (Peng et al., 2023):
      f_i  = theta^(-2i/dim), i < dim/2
      c(b) = dim * ln(L_orig / (2 pi b)) / (2 ln theta)   (dimension whose
             wavelength makes b rotations over the original context)
      low  = max(floor(c(beta_fast)), 0), high = min(ceil(c(beta_slow)), dim-1)
      ramp = clamp((i - low) / (high - low), 0, 1)   (high - low bumped by 1e-3 if 0)
      f'_i = f_i / factor * ramp + f_i * (1 - ramp)
    Precision reading: f'_i in f64 then rounded to f32; angle = f32(pos) * f'_i
    rounded in f32; cos and sin of that f32 angle in f64, rounded to f32.
    """
    half = rope_dim // 2
    i = np.arange(half, dtype=np.float64)
    freqs = theta ** (-2.0 * i / rope_dim)
    if original_seq_len > 0:
        def correction_dim(rotations):
            return rope_dim * math.log(original_seq_len / (rotations * 2 * math.pi)) / (2 * math.log(theta))
        low = max(math.floor(correction_dim(beta_fast)), 0)
        high = min(math.ceil(correction_dim(beta_slow)), rope_dim - 1)
        span = (high - low) if high != low else 0.001
        ramp = np.clip((i - low) / span, 0.0, 1.0)
        freqs = freqs / factor * ramp + freqs * (1.0 - ramp)
    f32 = freqs.astype(np.float32)
    pos = np.arange(max_pos, dtype=np.float32)
    angle = pos[:, None] * f32[None, :]                  # float32 * float32 -> float32
    a64 = angle.astype(np.float64)
    return np.cos(a64).astype(np.float32), np.sin(a64).astype(np.float32)


# ----------------------------------------------------------------------------- key path
def linear_bf16(x_bits: np.ndarray, w_bits: np.ndarray) -> np.ndarray:
    """bf16 Linear y = x W^T with no bias (index-keys page, Indexer.__init__: wk is a
    bf16 Linear(head_dim -> index_head_dim)). Reading: the sum of products is taken
    exactly (f64 accumulation of exact bf16*bf16 products) and rounded once to bf16."""
    x = bf16_to_f64(x_bits)
    w = bf16_to_f64(w_bits)
    return f64_to_bf16(x @ w.T)


def rmsnorm_bf16(x_bits: np.ndarray, w_bits: np.ndarray, eps: float) -> np.ndarray:
    """RMSNorm(index_head_dim, norm_eps) of the index keys (index-keys page,
    Indexer.__init__ / forward: k = k_norm(wk(latent))). The body is not on the
    pages. Reading: y_i = bf16( (w_i * x_i) * (1 / sqrt(mean_j x_j^2 + eps)) ),
    evaluated in f64 with eps taken as the f32 value of norm_eps."""
    x = bf16_to_f64(x_bits)
    w = bf16_to_f64(w_bits)
    ms = np.sum(x * x, axis=-1, keepdims=True) / x.shape[-1]
    r = 1.0 / np.sqrt(ms + float(np.float32(eps)))
    return f64_to_bf16((w * x) * r)


def rope_interleaved(x_bits: np.ndarray, cos: np.ndarray, sin: np.ndarray, positions: np.ndarray,
                     rope_dim: int) -> np.ndarray:
    """apply_rotary_emb on the last rope_dim dims (index-keys page, Indexer.forward:
    apply_rotary_emb(k[..., -rd:], freqs) and the same on q). The body is not on
    the pages. Reading: the complex view pairs dims (2i, 2i+1) of the rope slice
    and multiplies by table entry i of the row's position, in f32:
        y0 = f32(f32(x0*c) - f32(x1*s)),  y1 = f32(f32(x0*s) + f32(x1*c)),
    then rounds to bf16 (the tensor is bf16 and is rotated in place).
    x_bits: [..., D]; positions: broadcastable to x_bits.shape[:-1]."""
    x_bits = np.array(x_bits, dtype=np.uint16, copy=True)
    D = x_bits.shape[-1]
    r = bf16_to_f64(x_bits[..., D - rope_dim:]).astype(np.float32)
    x0 = r[..., 0::2]
    x1 = r[..., 1::2]
    pos = np.broadcast_to(np.asarray(positions), x_bits.shape[:-1])
    c = cos[pos]
    s = sin[pos]
    y0 = (x0 * c) - (x1 * s)
    y1 = (x0 * s) + (x1 * c)
    y = np.empty_like(r)
    y[..., 0::2] = y0
    y[..., 1::2] = y1
    x_bits[..., D - rope_dim:] = f32_to_bf16(y)
    return x_bits


def _e8m0_exponent(amax: np.ndarray) -> np.ndarray:
    """Smallest integer e with 6 * 2**e >= max(amax, 6 * 2**-126): the power-of-two
    ceiling of amax / 6 with amax floored at 6 * 2**-126 (compress module page,
    fp4_quant_e8m0_inplace)."""
    a = np.maximum(amax, SCALE_FLOOR)
    e = np.ceil(np.log2(a / 6.0)).astype(np.int64)      # first guess, then made exact
    e = np.where(np.ldexp(6.0, e - 1) >= a, e - 1, e)
    e = np.where(np.ldexp(6.0, e) < a, e + 1, e)
    return e


def fp4_quant_e8m0(x_bits: np.ndarray, block: int = FP4_BLOCK):
    """fp4_act_quant(x, block, inplace=True) with e8m0 scales (index-keys page,
    Indexer.forward; compress module page, fp4_quant_e8m0_inplace / to_e2m1_rne):
    per block of 32, scale = 2**e with e the pow2 ceiling of amax/6 (amax floored
    at 6*2**-126); values x / scale rounded onto the e2m1 grid to nearest, ties
    to the even code, keeping the sign.

    Returns (codes uint8 [..., n] with sign in bit 3, scale bytes uint8 [..., n/32]
    = e + 127, dequantised f64 values [..., n])."""
    x_bits = np.asarray(x_bits, dtype=np.uint16)
    shp = x_bits.shape
    nb = shp[-1] // block
    x = bf16_to_f64(x_bits).reshape(*shp[:-1], nb, block)
    neg = ((x_bits >> 15) & 1).reshape(*shp[:-1], nb, block).astype(np.uint8)
    e = _e8m0_exponent(np.max(np.abs(x), axis=-1))
    y = np.ldexp(np.abs(x), -e[..., None])                     # exact
    dist = np.abs(y[..., None] - E2M1_GRID)                    # [..., nb, 32, 8]
    best = dist.min(axis=-1, keepdims=True)
    is_best = dist == best
    # among (at most two, adjacent) nearest grid points take the even code
    even = (np.arange(8) % 2 == 0)
    choose_even = is_best & even
    mag = np.where(choose_even.any(axis=-1), np.argmax(choose_even, axis=-1), np.argmax(is_best, axis=-1))
    codes = (mag.astype(np.uint8) | (neg << 3)).reshape(shp)
    scales = (e + 127).astype(np.uint8)
    deq = (np.where(neg == 1, -1.0, 1.0) * np.ldexp(E2M1_GRID[mag], e[..., None])).reshape(shp)
    return codes, scales, deq


def pack_row68(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """The MXFP4 cache row (attention.py patch page, _indexer_k_cache_head_dim):
    64 bytes of packed e2m1 then 4 UE8M0 scale bytes. Packing reading: element
    2i in the low nibble of byte i, element 2i+1 in the high nibble; scale byte j
    belongs to block j (elements 32j .. 32j+31)."""
    lo = codes[..., 0::2].astype(np.uint8)
    hi = codes[..., 1::2].astype(np.uint8)
    return np.concatenate([lo | (hi << 4), scales.astype(np.uint8)], axis=-1)


def unpack_row68(rows: np.ndarray, head_dim: int = 128):
    rows = np.asarray(rows, dtype=np.uint8)
    nbytes = head_dim // 2
    packed = rows[..., :nbytes]
    codes = np.empty(rows.shape[:-1] + (head_dim,), dtype=np.uint8)
    codes[..., 0::2] = packed & 0xF
    codes[..., 1::2] = packed >> 4
    return codes, rows[..., nbytes:nbytes + head_dim // FP4_BLOCK]


def dequant_row68(rows: np.ndarray, head_dim: int = 128) -> np.ndarray:
    """Exact f64 values of packed rows: sign * grid[mag] * 2**(scale_byte - 127)."""
    codes, scales = unpack_row68(rows, head_dim)
    mag = E2M1_GRID[codes & 7]
    sign = np.where(codes & 8, -1.0, 1.0)
    e = scales.astype(np.int64) - 127
    e_full = np.repeat(e, FP4_BLOCK, axis=-1)
    return sign * np.ldexp(mag, e_full)


# ----------------------------------------------------------------------------- FP8 rows
# The FP8 indexer cache row (attention.py patch page, _indexer_k_cache_head_dim, FP8
# branch: "128 fp8 + 4 fp32 scale" = 132 bytes for head_dim 128; DeepseekV4Indexer:
# scale_fmt "ue8m0", quant_block_size 128). Readings: one block of 128 values per
# row; the scale is a power of two (UE8M0), the ceiling of amax / 448 (448 = largest
# e4m3 magnitude) with amax floored at 448 * 2**-126, stored as an f32; values x / scale
# rounded to the nearest e4m3 value, ties to the even code, keeping the sign; codes
# element i in byte i, then the f32 scale (little-endian).
FP8_BLOCK = 128
FP8_MAX = 448.0
FP8_SCALE_FLOOR = FP8_MAX * 2.0 ** -126
FP8_ROW_BYTES = 128 + 4
# e4m3 (the OCP "fn" variant: no infinities, code 0x7F is NaN) magnitudes by 7-bit code:
# exponent field E = code >> 3, mantissa M = code & 7; E = 0: M/8 * 2**-6 (subnormal),
# else (1 + M/8) * 2**(E - 7). Codes 0..126 ascend.
E4M3_GRID = np.array([((c & 7) / 8.0) * 2.0 ** -6 if (c >> 3) == 0 else (1.0 + (c & 7) / 8.0) * 2.0 ** ((c >> 3) - 7)
                      for c in range(127)])


def _ue8m0_exponent_fp8(amax: np.ndarray) -> np.ndarray:
    """Smallest integer e with 448 * 2**e >= max(amax, 448 * 2**-126)."""
    a = np.maximum(amax, FP8_SCALE_FLOOR)
    e = np.ceil(np.log2(a / FP8_MAX)).astype(np.int64)   # first guess, then made exact
    e = np.where(np.ldexp(FP8_MAX, e - 1) >= a, e - 1, e)
    e = np.where(np.ldexp(FP8_MAX, e) < a, e + 1, e)
    return e


def fp8_quant_ue8m0(x_bits: np.ndarray):
    """Per 128-value row: scale 2**e (e from _ue8m0_exponent_fp8 of the row's amax),
    x / 2**e (exact) rounded to the nearest e4m3 magnitude, ties to the even code,
    sign in bit 7. Returns (codes uint8 [..., 128], exponents int64 [...], dequantised
    f64 values [..., 128])."""
    x_bits = np.asarray(x_bits, dtype=np.uint16)
    x = bf16_to_f64(x_bits)
    neg = ((x_bits >> 15) & 1).astype(np.uint8)
    e = _ue8m0_exponent_fp8(np.max(np.abs(x), axis=-1))
    y = np.ldexp(np.abs(x), -e[..., None])                   # exact, <= 448
    hi = np.clip(np.searchsorted(E4M3_GRID, y, side="left"), 0, len(E4M3_GRID) - 1)
    lo = np.maximum(hi - 1, 0)
    d_hi, d_lo = E4M3_GRID[hi] - y, y - E4M3_GRID[lo]
    take_lo = (d_lo < d_hi) | ((d_lo == d_hi) & (lo % 2 == 0))
    mag = np.where(take_lo, lo, hi).astype(np.uint8)
    codes = mag | (neg << 7)
    deq = np.where(neg == 1, -1.0, 1.0) * np.ldexp(E4M3_GRID[mag], e[..., None])
    return codes, e, deq


def pack_row132(codes: np.ndarray, e: np.ndarray) -> np.ndarray:
    """128 code bytes then the f32 scale 2**e, little-endian."""
    sc = np.ldexp(np.ones(e.shape, dtype=np.float32), e.astype(np.int32)).astype("<f4")
    return np.concatenate([codes.astype(np.uint8), sc[..., None].view(np.uint8)], axis=-1)


def dequant_row132(rows: np.ndarray) -> np.ndarray:
    """Exact f64 values of FP8 rows: sign * e4m3 magnitude * scale."""
    rows = np.asarray(rows, dtype=np.uint8)
    codes = rows[..., :128]
    sc = np.ascontiguousarray(rows[..., 128:132]).view("<f4")[..., 0].astype(np.float64)
    mag = E4M3_GRID[np.minimum(codes & 0x7F, 126)]
    return np.where(codes & 0x80, -1.0, 1.0) * mag * sc[..., None]


def dequant_row(rows: np.ndarray) -> np.ndarray:
    """Dequantised values of 68-byte (MXFP4) or 132-byte (FP8) rows."""
    return dequant_row132(rows) if rows.shape[-1] == FP8_ROW_BYTES else dequant_row68(rows)


def quantise_rows(x_bits: np.ndarray, fmt: str = "mxfp4") -> np.ndarray:
    """The cache row of each 128-value vector in the given format."""
    if fmt == "fp8":
        codes, e, _ = fp8_quant_ue8m0(x_bits)
        return pack_row132(codes, e)
    codes, scales, _ = fp4_quant_e8m0(x_bits)
    return pack_row68(codes, scales)


def key_slots(start_pos: int, G: int, ratio: int):
    """Cache slots and RoPE positions of the G keys published by one forward
    (index-keys page, Indexer.forward, key publish): prefill (start_pos == 0)
    publishes groups 0..G-1, group j at position j*ratio; decode publishes the
    one group completed at start_pos into slot start_pos // ratio at position
    start_pos + 1 - ratio. In both cases slot s sits at position s * ratio."""
    if start_pos == 0:
        slots = np.arange(G)
        return slots, slots * ratio
    if G != 1 or (start_pos + 1) % ratio != 0:
        raise ValueError("decode publishes one key, on the token that completes a group")
    return np.array([start_pos // ratio]), np.array([start_pos + 1 - ratio])


def publish_keys(latent_bits, wk_bits, knorm_bits, cos, sin, start_pos: int, ratio: int,
                 rope_dim: int, eps: float, fmt: str = "mxfp4"):
    """Key publish (index-keys page, Indexer.forward): k = k_norm(wk(latent)),
    RoPE on the last rope_dim dims at the group position, fp4_act_quant, and the
    row written at slot start_pos//ratio + j. Returns (slots, rows [B, G, 68],
    bf16 keys before quantisation [B, G, D])."""
    B, G, _ = latent_bits.shape
    slots, positions = key_slots(start_pos, G, ratio)
    k = linear_bf16(latent_bits, wk_bits)
    k = rmsnorm_bf16(k, knorm_bits, eps)
    k = rope_interleaved(k, cos, sin, positions[None, :], rope_dim)
    return slots, quantise_rows(k, fmt), k


def project_queries(qr_bits: np.ndarray, wq_b_bits: np.ndarray, n_heads: int) -> np.ndarray:
    """q = wq_b(qr) unflattened to [..., n_heads, 128] (index-keys page, Indexer.forward:
    self.wq_b(qr).unflatten(-1, (n_local_heads, index_head_dim))). Reading: wq_b is a bf16
    Linear with no bias, its sum taken exactly and rounded once to bf16 (linear_bf16).
    qr_bits [..., Kq]; wq_b_bits [n_heads * 128, Kq]."""
    q = linear_bf16(qr_bits, wq_b_bits)
    return q.reshape(*q.shape[:-1], n_heads, q.shape[-1] // n_heads)


def prep_queries(q_bits, w_bits, cos, sin, start_pos: int, rope_dim: int, n_heads: int,
                 row_positions: Optional[np.ndarray] = None, fmt: str = "mxfp4"):
    """Query prep (index-keys page, Indexer.forward and __init__): RoPE at the
    query's own position start_pos + s, fp4_act_quant, and head weights scaled by
    softmax_scale * n_heads**-0.5 with softmax_scale = index_head_dim**-0.5.
    Reading: the weight product is kept in f64 (not rounded to bf16).
    q_bits [B, S, H, D]; w_bits [B, S, H]; row_positions overrides the
    positions of the S rows (used for sampled rows). Returns (rows [B,S,H,68],
    w' f64 [B,S,H], bf16 q after RoPE)."""
    B, S, H, D = q_bits.shape
    pos = (start_pos + np.arange(S)) if row_positions is None else np.asarray(row_positions)
    qr = rope_interleaved(q_bits, cos, sin, np.broadcast_to(pos[None, :, None], (B, S, H)), rope_dim)
    # softmax_scale * n_heads**-0.5 = (D * H)**-0.5, evaluated with one rounding (exact
    # whenever D * H is a power of four)
    wprime = bf16_to_f64(w_bits) * (float(D * n_heads) ** -0.5)
    return quantise_rows(qr, fmt), wprime, qr


def visible_lens(start_pos: int, S: int, ratio: int, row_positions: Optional[np.ndarray] = None):
    """compress_lens per query row (index-keys page, Indexer.forward, causal
    mask): prefill rows see (s + 1) // ratio keys, a decode row end_pos // ratio;
    both are (position + 1) // ratio."""
    pos = (start_pos + np.arange(S)) if row_positions is None else np.asarray(row_positions)
    return (pos + 1) // ratio


def index_scores(q_rows, wprime, k_rows, T: int, vis: np.ndarray, chunk: int = 256):
    """score[b,s,t] = sum_h w'[b,s,h] * relu(sum_d q[b,s,h,d] * k[b,t,d]) over the
    dequantised fp4 values (index-keys page, Indexer.forward: einsum bshd,btd->bsht,
    relu, times weights, sum over heads), with t >= vis[s] set to -inf (causal
    mask). f64 throughout; q rows [B,S,H,68 or 132], k rows [B,>=T,same width], vis [S]."""
    B, S, H, _ = q_rows.shape
    kd = dequant_row(k_rows[:, :T])                         # [B, T, D]
    out = np.empty((B, S, T), dtype=np.float64)
    t = np.arange(T)
    for b in range(B):
        for s0 in range(0, S, chunk):
            s1 = min(S, s0 + chunk)
            qd = dequant_row(q_rows[b, s0:s1])              # [s, H, D]
            dots = np.einsum("shd,td->sht", qd, kd[b])
            sc = np.einsum("sht,sh->st", np.maximum(dots, 0.0), wprime[b, s0:s1])
            sc[t[None, :] >= vis[s0:s1, None]] = -np.inf
            out[b, s0:s1] = sc
    return out


# ----------------------------------------------------------------------------- selection
def select_candidate_blocks(scores: np.ndarray, vis: np.ndarray, cand_topk_blocks: int,
                            cand_block_size: int) -> np.ndarray:
    """Level one of the two-level top-k (compress module page, select_candidate_blocks:
    logits[queries][width] with unreachable positions at -inf and compress_lens[q]
    in, keep mask [queries][width] out; index-keys page, Indexer.forward).

    The body is not on the pages ("parity unpinned" for this reading). Reading:
    blocks are [j*cbs, (j+1)*cbs) (the last may be partial); a block is eligible
    when it holds a reachable position (j*cbs < compress_len); its score is the
    max of its finite logits; the cand_topk_blocks best eligible blocks are kept,
    ties to the lower block index. Returns kept block ids [R, cbk] ascending,
    padded with -1 (the keep mask is every position of a kept block)."""
    R, T = scores.shape
    nblk = -(-T // cand_block_size)
    out = np.full((R, cand_topk_blocks), -1, dtype=np.int32)
    for r in range(R):
        cands = []
        for j in range(nblk):
            lo, hi = j * cand_block_size, min((j + 1) * cand_block_size, T)
            if lo >= vis[r]:
                continue
            blk = scores[r, lo:hi]
            finite = blk[np.isfinite(blk)]
            if finite.size == 0:
                continue
            cands.append((-finite.max(), j))
        cands.sort()
        kept = sorted(j for _, j in cands[:cand_topk_blocks])
        out[r, :len(kept)] = kept
    return out


def candidate_mask(blocks: np.ndarray, T: int, cand_block_size: int) -> np.ndarray:
    """Keep mask [R, T] of the kept block ids (-1 entries ignored)."""
    R = blocks.shape[0]
    keep = np.zeros((R, T), dtype=bool)
    for r in range(R):
        for j in blocks[r]:
            if j >= 0:
                keep[r, j * cand_block_size:min((j + 1) * cand_block_size, T)] = True
    return keep


def topk_positions(scores: np.ndarray, vis: np.ndarray, index_topk: int, offset: int, T: int) -> np.ndarray:
    """Top-k, re-sorted into position order, offset added, -1 where unreachable
    (index-keys page, Indexer.forward, final three lines; attention.py patch page,
    _fill_short_context_topk_indices for the -1 padding to the full TOP_K width).

    k_eff = min(index_topk, T). Among the row's finite scores at positions
    t < vis, keep the k_eff largest, ties to the lower position; emit them in
    ascending position order as t + offset, then -1 up to index_topk columns.
    Reading: a -inf score (masked by the candidate filter) is never emitted.
    With no candidate filter and vis <= k_eff this is exactly [0 .. vis) then -1,
    the short-context fill. scores [R, T]; returns int32 [R, index_topk]."""
    R = scores.shape[0]
    k_eff = min(index_topk, T)
    out = np.full((R, index_topk), -1, dtype=np.int32)
    for r in range(R):
        v = int(min(vis[r], T))
        row = scores[r, :v]
        cand = np.nonzero(np.isfinite(row))[0]
        if cand.size > k_eff:
            order = np.lexsort((cand, -row[cand]))          # score desc, then position asc
            cand = np.sort(cand[order[:k_eff]])
        out[r, :cand.size] = cand + offset
    return out


def forward(q_bits, w_bits, k_rows, cos, sin, start_pos: int, ratio: int, rope_dim: int, index_topk: int,
            offset: int, cand_in: Optional[np.ndarray] = None, cand_topk_blocks: int = 0,
            cand_block_size: int = 0, want_candidates: bool = False, fmt: Optional[str] = None):
    """Indexer.forward after the key publish (index-keys page): query prep,
    scores, causal mask, optional level-one candidate publication (source layer)
    or level-two candidate mask (consumer), then top-k. k_rows is the cache
    after this forward's keys were published. Returns (topk int32 [B,S,k],
    candidate blocks [B,S,cbk] or None, masked scores [B,S,T])."""
    B, S, H, D = q_bits.shape
    T = (start_pos + S) // ratio
    if fmt is None:   # the queries take the keys' format
        fmt = "fp8" if k_rows.shape[-1] == FP8_ROW_BYTES else "mxfp4"
    q_rows, wprime, _ = prep_queries(q_bits, w_bits, cos, sin, start_pos, rope_dim, H, fmt=fmt)
    vis = visible_lens(start_pos, S, ratio)
    sc = index_scores(q_rows, wprime, k_rows, T, vis)
    cand_out = None
    flat = sc.reshape(B * S, T)
    vis_flat = np.tile(vis, B)
    if want_candidates:
        cand_out = select_candidate_blocks(flat, vis_flat, cand_topk_blocks, cand_block_size).reshape(B, S, -1)
    if cand_in is not None:
        keep = candidate_mask(cand_in.reshape(B * S, -1), T, cand_block_size)
        flat = np.where(keep, flat, -np.inf)
        sc = flat.reshape(B, S, T)
    top = topk_positions(flat, vis_flat, index_topk, offset, T).reshape(B, S, index_topk)
    return top, cand_out, sc


# ----------------------------------------------------------------------------- upstream producers
# The inputs of the key publish and the query prep come from three producers on the pages:
# the Compressor's latent (compress module page, compressor / Compressor.forward; attention.py
# patch page, compressor_kv_score and fused_wkv_wgate), the head weights (index-keys page,
# Indexer.__init__ weights_proj, Indexer.forward weights line), and the fp4 quantiser with
# e4m3 scales that the compressed latent goes through (compress module page,
# fp4_quant_e4m3_inplace, LATENT_BLOCK, precision policy).

# Block size of the compressed latent's quantiser (compress module page, LATENT_BLOCK:
# fp4_act_quant(latent, 16, ...)) and its amax floor (fp4_quant_e4m3_inplace: 6 * 2^-9).
LATENT_BLOCK = 16
LATENT_SCALE_FLOOR = 6.0 * 2.0 ** -9


def e4m3_round(y: np.ndarray) -> np.ndarray:
    """Non-negative f64 values rounded to the nearest e4m3 ("fn" variant, largest 448)
    magnitude, ties to the even code, saturating at 448. Returns the 7-bit magnitude codes."""
    y = np.minimum(np.asarray(y, dtype=np.float64), E4M3_GRID[-1])
    hi = np.clip(np.searchsorted(E4M3_GRID, y, side="left"), 0, len(E4M3_GRID) - 1)
    lo = np.maximum(hi - 1, 0)
    d_hi, d_lo = E4M3_GRID[hi] - y, y - E4M3_GRID[lo]
    take_lo = (d_lo < d_hi) | ((d_lo == d_hi) & (lo % 2 == 0))
    return np.where(take_lo, lo, hi).astype(np.uint8)


def fp4_quant_e4m3(x_bits: np.ndarray, block: int = LATENT_BLOCK):
    """fp4_quant_e4m3_inplace (compress module page): per block of 16 values, amax floored at
    6 * 2^-9, scale = amax / 6 rounded through e4m3, values x / scale rounded onto the e2m1
    grid (to nearest, ties to the even code, keeping the sign; beyond 6 the nearest grid
    point is 6), dequantised back to bf16 (sign * grid * scale has at most 6 significant
    bits, so it is exact in bf16 down to the subnormal range). Readings: amax / 6 and
    x / scale are the exact quotients (f64 here; a quotient that sits on a tie is exactly
    representable, so f64 decides ties like exact arithmetic).
    Returns (codes uint8 [..., n] with sign in bit 3, scale magnitude codes uint8
    [..., n / 16] (e4m3, positive), dequantised bf16 bits [..., n])."""
    x_bits = np.asarray(x_bits, dtype=np.uint16)
    shp = x_bits.shape
    nb = shp[-1] // block
    x = bf16_to_f64(x_bits).reshape(*shp[:-1], nb, block)
    neg = ((x_bits >> 15) & 1).reshape(*shp[:-1], nb, block).astype(np.uint8)
    amax = np.maximum(np.max(np.abs(x), axis=-1), LATENT_SCALE_FLOOR)
    sc_code = e4m3_round(amax / 6.0)
    sc = E4M3_GRID[sc_code]
    y = np.abs(x) / sc[..., None]
    dist = np.abs(y[..., None] - E2M1_GRID)
    best = dist.min(axis=-1, keepdims=True)
    is_best = dist == best
    even = (np.arange(8) % 2 == 0)
    choose_even = is_best & even
    mag = np.where(choose_even.any(axis=-1), np.argmax(choose_even, axis=-1), np.argmax(is_best, axis=-1))
    codes = (mag.astype(np.uint8) | (neg << 3)).reshape(shp)
    deq = np.where(neg == 1, -1.0, 1.0) * E2M1_GRID[mag] * sc[..., None]
    return codes, sc_code, f64_to_bf16(deq.reshape(shp))


def weights_proj(x_bits: np.ndarray, wp_bits: np.ndarray) -> np.ndarray:
    """w = weights_proj(x) (index-keys page, Indexer.__init__: weights_proj is a bf16 Linear
    dim -> n_heads; Indexer.forward: weights = weights_proj(x) * ...). Reading: no bias, the
    exact sum rounded once to bf16, as linear_bf16. x_bits [..., dim]; wp_bits [n_heads, dim]."""
    return linear_bf16(x_bits, wp_bits)


def compress_latent(x_bits: np.ndarray, wkv_bits: np.ndarray, wgate_bits: np.ndarray, norm_bits: np.ndarray,
                    ratio: int, eps: float) -> np.ndarray:
    """Compressor.forward (compress module page: softmax pooling of ratio tokens into one
    latent, a plain projection at ratio 1; the compressor is f32 until its RMSNorm casts to
    bf16; attention.py patch page: kv_score = hidden_states @ fused_wkv_wgate.weight^T with
    an f32 result). Readings, where the pages give no body:
      kv[t] = x[t] Wkv^T and score[t] = x[t] Wgate^T (the two halves of fused_wkv_wgate),
        as exact sums (the GPU accumulates in f32);
      group g holds tokens g*ratio .. g*ratio + ratio - 1 of the sequence; per latent dim d,
        the weights are the softmax over those tokens of score[., d], and the pooled value is
        sum_t softmax_t * kv[t, d] (at ratio 1 the softmax is 1: the plain projection);
      RMSNorm of the pooled vector as rmsnorm_bf16 reads it (bf16((w * p) / sqrt(mean(p^2) +
        eps))), on the unrounded pooled values.
    x_bits [B, S, dim] bf16 with S a multiple of ratio; wkv_bits, wgate_bits [hd, dim];
    norm_bits [hd]. Returns the latent bf16 bits [B, S / ratio, hd]."""
    x = bf16_to_f64(x_bits)
    kv = x @ bf16_to_f64(wkv_bits).T
    sc = x @ bf16_to_f64(wgate_bits).T
    B, S, hd = kv.shape
    G = S // ratio
    kv = kv[:, :G * ratio].reshape(B, G, ratio, hd)
    sc = sc[:, :G * ratio].reshape(B, G, ratio, hd)
    e = np.exp(sc - sc.max(axis=2, keepdims=True))
    pooled = (e * kv).sum(axis=2) / e.sum(axis=2)
    ms = np.sum(pooled * pooled, axis=-1, keepdims=True) / hd
    r = 1.0 / np.sqrt(ms + float(np.float32(eps)))
    return f64_to_bf16((bf16_to_f64(norm_bits) * pooled) * r)
