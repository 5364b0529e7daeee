"""Seeded synthetic inputs for the indexer workloads.

This module is shared by the oracle-side tests, the GPU parity tests and the
benchmark. It holds NONE of the indexer's arithmetic: only workload shapes and
a counter-based random-number generator (splitmix64 -> Box-Muller) that turns
(seed, tensor name, flat element index) into a bf16 value. Because every
element depends only on its own index, any slice of a tensor (a few sampled
query rows, say) can be generated on its own and agrees with the full tensor.

splitmix64 is Vigna's published 64-bit mixer (golden-gamma increment
0x9E3779B97F4A7C15 followed by the two xor-shift-multiply rounds). The
Box-Muller transform maps two uniforms in (0, 1] to one N(0, 1) draw.
f64 draws are rounded to f32 and then to bf16 (both round-to-nearest-even);
the generator only has to be deterministic, so this double rounding is fine.

All arithmetic runs in torch so that large tensors can be generated directly
on the GPU; int64 multiplication wraps modulo 2**64 exactly like uint64.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

__all__ = [
    "Workload",
    "WORKLOADS",
    "RopeParams",
    "ROPE",
    "stream_id",
    "uniform_flat",
    "normal_bf16_flat",
    "normal_bf16",
    "uniform_f64",
]

_MASK64 = (1 << 64) - 1


def _s64(x: int) -> int:
    """Two's-complement view of a 64-bit unsigned constant (torch has no uint64 math)."""
    x &= _MASK64
    return x - (1 << 64) if x >= (1 << 63) else x


_GAMMA = _s64(0x9E3779B97F4A7C15)
_M1 = _s64(0xBF58476D1CE4E5B9)
_M2 = _s64(0x94D049BB133111EB)


def _srl(x: torch.Tensor, k: int) -> torch.Tensor:
    """Logical right shift of int64 bit patterns."""
    return (x >> k) & ((1 << (64 - k)) - 1)


def _mix(z: torch.Tensor) -> torch.Tensor:
    z = (z ^ _srl(z, 30)) * _M1
    z = (z ^ _srl(z, 27)) * _M2
    return z ^ _srl(z, 31)


def _mix_int(z: int) -> int:
    z &= _MASK64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _MASK64
    return z ^ (z >> 31)


def stream_id(seed: int, name: str) -> int:
    """64-bit stream key for one named tensor (FNV-1a of the name, mixed with the seed)."""
    h = 0xCBF29CE484222325
    for ch in name.encode():
        h = ((h ^ ch) * 0x100000001B3) & _MASK64
    return _mix_int(h ^ _mix_int(seed + 0x5DEECE66D))


def _raw64(stream: int, counters: torch.Tensor) -> torch.Tensor:
    """splitmix64 output for state = stream + (counter + 1) * gamma."""
    state = counters * _GAMMA + _s64(stream + 0x9E3779B97F4A7C15)
    return _mix(state)


def uniform_flat(stream: int, start: int, count: int, device="cpu") -> torch.Tensor:
    """f64 uniforms in (0, 1] for counters [start, start + count)."""
    c = torch.arange(start, start + count, dtype=torch.int64, device=device)
    z = _raw64(stream, c)
    return (_srl(z, 11).to(torch.float64) + 1.0) * (2.0 ** -53)


def normal_bf16_flat(stream: int, start: int, count: int, std: float = 1.0,
                     mean: float = 0.0, device="cpu") -> torch.Tensor:
    """bf16 N(mean, std^2) draws for flat element indices [start, start + count).

    Element i uses the uniforms at counters 2i and 2i + 1 of the stream.
    """
    c = torch.arange(2 * start, 2 * (start + count), dtype=torch.int64, device=device)
    z = _raw64(stream, c).view(count, 2)
    u = (_srl(z, 11).to(torch.float64) + 1.0) * (2.0 ** -53)
    n = torch.sqrt(-2.0 * torch.log(u[:, 0])) * torch.cos((2.0 * math.pi) * u[:, 1])
    return (n * std + mean).to(torch.float32).to(torch.bfloat16)


def normal_bf16(seed: int, name: str, shape, std: float = 1.0, mean: float = 0.0,
                device="cpu", chunk: int = 1 << 24) -> torch.Tensor:
    """A whole bf16 tensor of the given shape, generated in chunks."""
    n = int(math.prod(shape))
    out = torch.empty(n, dtype=torch.bfloat16, device=device)
    sid = stream_id(seed, name)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        out[s:e] = normal_bf16_flat(sid, s, e - s, std, mean, device)
    return out.view(*shape)


def uniform_f64(seed: int, name: str, shape, device="cpu") -> torch.Tensor:
    n = int(math.prod(shape))
    return uniform_flat(stream_id(seed, name), 0, n, device).view(*shape)


@dataclasses.dataclass(frozen=True)
class RopeParams:
    """YaRN parameters of the compressed layers (theta is compress_rope_theta)."""
    theta: float = 160000.0
    factor: float = 16.0
    original_seq_len: int = 4096
    beta_fast: float = 32.0
    beta_slow: float = 1.0


ROPE = RopeParams()


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic indexer workload: shapes, positions and selection sizes.

    Sizes follow the five workloads the indexer is exercised on: a tiny
    prefill, a 32-sequence decode over 8192 compressed positions, an 8192-row
    prefill, a two-level long-context decode and a 65536-row top-k-heavy
    prefill.
    """
    name: str
    B: int
    S: int
    start_pos: int
    ratio: int
    H: int
    topk: int
    offset: int = 0
    D: int = 128
    rope_dim: int = 64
    cand_topk_blocks: int = 0
    cand_block_size: int = 0
    heavy_frac: float = 0.0
    heavy_scale: float = 1.0
    norm_eps: float = 1e-6
    seed: int = 0
    key_format: int = 0       # 0: MXFP4 rows (68 bytes), 1: FP8 rows (132 bytes)
    q_lora_rank: int = 1280   # K of the query projection wq_b (qr -> H * 128)
    fused_q: bool = False     # queries enter as qr: the projection wq_b runs inside the step
    dim: int = 4096           # hidden size of x for the upstream producers (not given on the pages)

    @property
    def end_pos(self) -> int:
        return self.start_pos + self.S

    @property
    def T(self) -> int:
        """Key width end_pos // ratio."""
        return self.end_pos // self.ratio

    @property
    def decode(self) -> bool:
        return self.start_pos > 0

    @property
    def two_level(self) -> bool:
        return self.cand_topk_blocks > 0

    @property
    def T_cap(self) -> int:
        """Cache capacity in keys (a multiple of 128)."""
        return (self.T + 127) // 128 * 128

    @property
    def max_pos(self) -> int:
        """Rows of the RoPE table needed (query positions reach end_pos - 1)."""
        return self.end_pos

    # ------------------------------------------------------------------ inputs
    def q(self, device="cpu", tag: str = "q") -> torch.Tensor:
        return normal_bf16(self.seed, f"{self.name}/{tag}", (self.B, self.S, self.H, self.D), device=device)

    def q_rows(self, rows, device="cpu", tag: str = "q") -> torch.Tensor:
        """Only the listed flat query rows (b * S + s) of q, [len(rows), H, D]."""
        sid = stream_id(self.seed, f"{self.name}/{tag}")
        per = self.H * self.D
        return torch.stack([normal_bf16_flat(sid, r * per, per, device=device).view(self.H, self.D)
                            for r in rows])

    def qr(self, device="cpu", tag: str = "qr") -> torch.Tensor:
        """The query latent fed to wq_b, [B, S, q_lora_rank] (unit normal)."""
        return normal_bf16(self.seed, f"{self.name}/{tag}", (self.B, self.S, self.q_lora_rank), device=device)

    def wq_b(self, device="cpu") -> torch.Tensor:
        """wq_b [H * 128, q_lora_rank], normal with std q_lora_rank^-0.5, so q has unit scale."""
        return normal_bf16(self.seed, f"{self.name}/wq_b", (self.H * self.D, self.q_lora_rank),
                           std=self.q_lora_rank ** -0.5, device=device)

    def w(self, device="cpu", tag: str = "w") -> torch.Tensor:
        w = normal_bf16(self.seed, f"{self.name}/{tag}", (self.B, self.S, self.H), device=device)
        if self.heavy_frac > 0:
            u = uniform_f64(self.seed, f"{self.name}/{tag}/heavy", (self.B, self.S), device=device)
            heavy = (u < self.heavy_frac).unsqueeze(-1)
            w = torch.where(heavy, (w.float() * self.heavy_scale).to(torch.bfloat16), w)
        return w

    def latent(self, device="cpu") -> torch.Tensor:
        """Latents that fill key slots 0 .. T-1 (the prefill-published keys)."""
        return normal_bf16(self.seed, f"{self.name}/latent", (self.B, self.T, self.D), device=device)

    def decode_latent(self, device="cpu") -> torch.Tensor:
        """The latent of the group completed at start_pos (decode publishes one key)."""
        return normal_bf16(self.seed, f"{self.name}/latent_step", (self.B, 1, self.D), device=device)

    def wk(self, device="cpu") -> torch.Tensor:
        return normal_bf16(self.seed, f"{self.name}/wk", (self.D, self.D), std=self.D ** -0.5, device=device)

    def k_norm_w(self, device="cpu") -> torch.Tensor:
        return normal_bf16(self.seed, f"{self.name}/k_norm_w", (self.D,), std=math.sqrt(0.1), mean=1.0,
                           device=device)

    # ------------------------------------------------------------ upstream producers
    def x(self, device="cpu") -> torch.Tensor:
        """Hidden states [B, S, dim] (unit normal) for the Compressor and weights_proj."""
        return normal_bf16(self.seed, f"{self.name}/x", (self.B, self.S, self.dim), device=device)

    def wkv(self, device="cpu") -> torch.Tensor:
        """Compressor kv projection [128, dim], std dim^-0.5 (kv of unit scale)."""
        return normal_bf16(self.seed, f"{self.name}/wkv", (self.D, self.dim), std=self.dim ** -0.5, device=device)

    def wgate(self, device="cpu") -> torch.Tensor:
        """Compressor gate projection [128, dim], std dim^-0.5."""
        return normal_bf16(self.seed, f"{self.name}/wgate", (self.D, self.dim), std=self.dim ** -0.5, device=device)

    def c_norm_w(self, device="cpu") -> torch.Tensor:
        """The Compressor's RMSNorm weight [128], 1 + N(0, 0.1) like k_norm."""
        return normal_bf16(self.seed, f"{self.name}/c_norm_w", (self.D,), std=math.sqrt(0.1), mean=1.0,
                           device=device)

    def wproj(self, device="cpu") -> torch.Tensor:
        """weights_proj [H, dim], std dim^-0.5 (head weights of unit scale)."""
        return normal_bf16(self.seed, f"{self.name}/wproj", (self.H, self.dim), std=self.dim ** -0.5, device=device)


WORKLOADS = {
    w.name: w
    for w in [
        Workload("tiny_prefill", B=1, S=256, start_pos=0, ratio=4, H=8, topk=16),
        Workload("decode", B=32, S=1, start_pos=32767, ratio=4, H=64, topk=2048),
        Workload("prefill", B=1, S=8192, start_pos=0, ratio=4, H=64, topk=512),
        Workload("two_level_decode", B=8, S=1, start_pos=131071, ratio=4, H=64, topk=2048,
                 cand_topk_blocks=64, cand_block_size=64),
        Workload("large_prefill", B=2, S=32768, start_pos=0, ratio=4, H=64, topk=2048, offset=8192,
                 heavy_frac=0.05, heavy_scale=8.0),
        # the FP8 key format (132-byte rows) on the decode and prefill shapes
        Workload("decode_fp8", B=32, S=1, start_pos=32767, ratio=4, H=64, topk=2048, key_format=1),
        Workload("prefill_fp8", B=1, S=8192, start_pos=0, ratio=4, H=64, topk=512, key_format=1),
        # the prefill shape with the query projection (qr -> wq_b -> q) fused into the query prep
        Workload("prefill_qproj", B=1, S=8192, start_pos=0, ratio=4, H=64, topk=512, fused_q=True),
    ]
}


@dataclasses.dataclass(frozen=True)
class MixedBatch:
    """A server batch: sequences with their own start position and query-row count (decode
    rows and prefill chunks), their keys in one shared pool of 64-key pages assigned in a
    seeded random order. Sequence b holds keys 0 .. T_b - 1 (key j published at RoPE
    position j * ratio, as a prefill publishes it) with T_b = (start_pos_b + S_b) // ratio;
    its rows are q_start[b] .. q_start[b+1] - 1 of the flat query batch."""
    name: str
    seqs: tuple            # ((start_pos, S), ...)
    ratio: int
    H: int
    topk: int
    offset: int = 0
    D: int = 128
    rope_dim: int = 64
    cand_topk_blocks: int = 0
    cand_block_size: int = 0
    spare_pages: int = 8   # pool pages no sequence owns
    norm_eps: float = 1e-6
    seed: int = 0
    key_format: int = 0       # 0: MXFP4 rows (68 bytes), 1: FP8 rows (132 bytes)

    @property
    def n_seq(self) -> int:
        return len(self.seqs)

    @property
    def Q(self) -> int:
        return sum(S for _, S in self.seqs)

    @property
    def q_start(self) -> list:
        out = [0]
        for _, S in self.seqs:
            out.append(out[-1] + S)
        return out

    @property
    def T_list(self) -> list:
        return [(sp + S) // self.ratio for sp, S in self.seqs]

    @property
    def T_max(self) -> int:
        return max(max(self.T_list), 1)

    @property
    def max_pos(self) -> int:
        return max(sp + S for sp, S in self.seqs)

    @property
    def pages(self) -> list:
        return [(t + 63) // 64 for t in self.T_list]

    @property
    def num_pages(self) -> int:
        return sum(self.pages) + self.spare_pages

    @property
    def bt_stride(self) -> int:
        return max((self.T_max + 63) // 64, 1)

    def block_table(self) -> torch.Tensor:
        """int32 [n_seq, bt_stride]: a seeded permutation of the pool's pages dealt to the
        sequences in order; unused entries -1."""
        u = uniform_f64(self.seed, f"{self.name}/pages", (self.num_pages,))
        perm = torch.argsort(u).to(torch.int32)
        bt = torch.full((self.n_seq, self.bt_stride), -1, dtype=torch.int32)
        k = 0
        for b, n in enumerate(self.pages):
            bt[b, :n] = perm[k:k + n]
            k += n
        return bt

    def q(self, device="cpu", tag: str = "q") -> torch.Tensor:
        return normal_bf16(self.seed, f"{self.name}/{tag}", (self.Q, self.H, self.D), device=device)

    def w(self, device="cpu", tag: str = "w") -> torch.Tensor:
        return normal_bf16(self.seed, f"{self.name}/{tag}", (self.Q, self.H), device=device)

    def latent(self, b: int, device="cpu") -> torch.Tensor:
        """Latents of sequence b's keys 0 .. T_b - 1, [T_b, D]."""
        return normal_bf16(self.seed, f"{self.name}/latent/{b}", (self.T_list[b], self.D), device=device)

    def wk(self, device="cpu") -> torch.Tensor:
        return normal_bf16(self.seed, f"{self.name}/wk", (self.D, self.D), std=self.D ** -0.5, device=device)

    def k_norm_w(self, device="cpu") -> torch.Tensor:
        return normal_bf16(self.seed, f"{self.name}/k_norm_w", (self.D,), std=math.sqrt(0.1), mean=1.0,
                           device=device)


def _server_step_seqs() -> tuple:
    """64 decode rows with context lengths spread over 4k .. 32k positions (each a group end,
    start_pos + 1 a multiple of 4) and two 512-row prefill chunks at 16384 and 24576."""
    u = uniform_f64(0, "server_step/lengths", (64,))
    dec = tuple((int(4096 + x * 28672) // 4 * 4 + 3, 1) for x in u.tolist())
    return dec + ((16384, 512), (24576, 512))


MIXED = {
    m.name: m
    for m in [
        # a small batch for parity: a chunked prefill, decode rows, a prefill from 0, an
        # empty sequence, a one-key sequence and a 2048-key sequence
        MixedBatch("mixed_small", seqs=((1024, 64), (4095, 1), (511, 1), (0, 40), (300, 0), (6, 1), (8191, 1)),
                   ratio=4, H=64, topk=128),
        # decode only (one row per sequence): the single-row score kernel over the pool
        MixedBatch("mixed_decode", seqs=tuple((4 * (256 + 97 * i) + 3, 1) for i in range(24)), ratio=4, H=64,
                   topk=256),
        # a server step: 64 decode rows + two 512-row prefill chunks
        MixedBatch("server_step", seqs=_server_step_seqs(), ratio=4, H=64, topk=2048),
    ]
}
