"""The seeded input generator: splitmix64 bits, slice consistency, shapes."""
import dataclasses
import math

import numpy as np
import torch

import workloads as W

MASK = (1 << 64) - 1


def _splitmix_ref(state):
    z = state & MASK
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK
    return z ^ (z >> 31)


def test_splitmix64_matches_integer_reference():
    sid = W.stream_id(0, "probe")
    c = torch.arange(0, 64, dtype=torch.int64)
    got = W._raw64(sid, c).numpy().view(np.uint64)
    for i in range(64):
        want = _splitmix_ref(sid + 0x9E3779B97F4A7C15 + i * 0x9E3779B97F4A7C15)
        assert int(got[i]) == want


def test_known_first_output_of_splitmix64():
    # Vigna's splitmix64 seeded with 0 yields 0xE220A8397B1DCDAF first.
    assert _splitmix_ref(0x9E3779B97F4A7C15) == 0xE220A8397B1DCDAF


def test_slices_agree_with_full_tensor():
    wl = W.WORKLOADS["tiny_prefill"]
    q = wl.q()
    rows = [0, 17, 255]
    sub = wl.q_rows(rows)
    for i, r in enumerate(rows):
        assert torch.equal(sub[i], q.view(-1, wl.H, wl.D)[r])


def test_normal_moments_and_determinism():
    x = W.normal_bf16(0, "moments", (200000,)).float()
    assert abs(x.mean().item()) < 0.01 and abs(x.std().item() - 1) < 0.01
    assert torch.equal(x, W.normal_bf16(0, "moments", (200000,)).float())
    assert not torch.equal(x, W.normal_bf16(1, "moments", (200000,)).float())


def test_workload_shapes():
    d = W.WORKLOADS["decode"]
    assert d.T == 8192 and d.decode and d.T_cap == 8192
    p = W.WORKLOADS["large_prefill"]
    assert p.T == 8192 and not p.decode and p.offset == 8192
    t = W.WORKLOADS["two_level_decode"]
    assert t.T == 32768 and t.two_level
    assert W.WORKLOADS["tiny_prefill"].T == 64


def test_heavy_rows_fraction():
    p = W.WORKLOADS["large_prefill"]
    u = W.uniform_f64(p.seed, f"{p.name}/w/heavy", (p.B, p.S))
    frac = (u < p.heavy_frac).double().mean().item()
    assert abs(frac - 0.05) < 0.005


def test_query_latent_and_projection_generators():
    """qr [B, S, q_lora_rank] is unit normal, wq_b [H * 128, q_lora_rank] has std
    q_lora_rank^-0.5 (so q = wq_b(qr) has unit scale), both deterministic and distinct."""
    wl = dataclasses.replace(W.WORKLOADS["prefill"], name="gen_qp", B=2, S=48, H=8, q_lora_rank=256)
    qr, wq = wl.qr(), wl.wq_b()
    assert qr.shape == (2, 48, 256) and wq.shape == (8 * 128, 256)
    assert qr.dtype == torch.bfloat16 and wq.dtype == torch.bfloat16
    assert torch.equal(qr, wl.qr()) and torch.equal(wq, wl.wq_b())
    assert abs(qr.float().std().item() - 1.0) < 0.05
    assert abs(wq.float().std().item() * 256 ** 0.5 - 1.0) < 0.05
    q = qr.float().reshape(-1, 256) @ wq.float().T
    assert 0.8 < q.std().item() < 1.2
    assert not torch.equal(qr, dataclasses.replace(wl, name="gen_qp2").qr())
