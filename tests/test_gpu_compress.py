"""GPU parity of the upstream producers (indexer_compress_weights: the Compressor's latent,
its fp4 / e4m3-scale quantised copy, and weights_proj) against the oracle, through the C ABI.

The kernel accumulates the projections in f32 on the tensor cores and pools in f32; the
oracle sums exactly and pools in f64, so a bf16 output may sit one unit away where the
exact value is within f32 rounding of a bf16 midpoint. Those are counted and bounded; the
quantised latent is decided in the kernel's precision from its own latent, so it is
compared bit for bit with the oracle's quantiser applied to that latent. Downstream, the
kernel's latent and head weights drive the key publish and the forward, which must match
the oracle run on the same latent and weights.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle as O
from tests import cases as C
from workloads import WORKLOADS

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def X():
    import sparse_attention_top_indexer_gb300 as X
    X.load_library()
    return X


def _ulps_apart(a_bits: np.ndarray, b_bits: np.ndarray) -> np.ndarray:
    """Distance in bf16 units between two arrays of bf16 bit patterns (same-sign ordering)."""
    def key(b):
        b = b.astype(np.int32)
        return np.where(b & 0x8000, -(b & 0x7FFF), b & 0x7FFF)
    return np.abs(key(a_bits) - key(b_bits))


def _run(X, wl, with_q=True):
    d = C.dims_of(wl)
    x, wkv, wg, nw, wp = wl.x("cuda"), wl.wkv("cuda"), wl.wgate("cuda"), wl.c_norm_w("cuda"), wl.wproj("cuda")
    G = wl.S // wl.ratio
    lat = torch.empty((wl.B, G, wl.D), dtype=torch.bfloat16, device="cuda")
    latq = torch.empty_like(lat) if with_q else None
    w = torch.empty((wl.B, wl.S, wl.H), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(X.STATUS_BYTES, dtype=torch.uint8, device="cuda")
    X.indexer_workspace_init(ws)
    X.indexer_compress_weights(d, x, wkv, wg, nw, wp, lat, w, ws, latent_q=latq)
    X.indexer_status(ws)
    return (x, wkv, wg, nw, wp), lat, latq, w


# cp_a: ratio 4, H 64, one ragged 128-row tile in K of 4 chunks; cp_b: 700 rows (six tiles),
# dim 4096; ratio 1, 2, 8, 16 and 32 (a group of 32 lanes: a whole warp); H 8 and 128
@pytest.mark.parametrize("name,B,S,ratio,H,dim", [
    ("cp_a", 1, 96, 4, 64, 256), ("cp_b", 2, 352, 4, 64, 4096), ("cp_r1", 1, 130, 1, 16, 512),
    ("cp_r2", 1, 64, 2, 8, 320), ("cp_r8", 1, 256, 8, 32, 192), ("cp_r16", 1, 160, 16, 128, 256),
    ("cp_r32", 3, 64, 32, 64, 128)])
def test_compress_weights_parity(X, name, B, S, ratio, H, dim):
    wl = dataclasses.replace(WORKLOADS["prefill"], name=name, B=B, S=S, ratio=ratio, H=H, dim=dim)
    (x, wkv, wg, nw, wp), lat, latq, w = _run(X, wl)
    xb = C.bits(x)
    # latent: the f32 sums carry an absolute error (about dim * 2^-24 * sum |x w| in kv and the
    # gate scores), which the pooling and the norm pass on; so a value may differ from the
    # exactly rounded one by one bf16 unit plus that absolute error, and rarely differs at all
    ref_lat = O.compress_latent(xb, C.bits(wkv), C.bits(wg), C.bits(nw), ratio, wl.norm_eps)
    got_lat = C.bits(lat)
    g64, r64 = O.bf16_to_f64(got_lat), O.bf16_to_f64(ref_lat)
    ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(r64), 2.0 ** -126))) - 7)
    rms = np.sqrt(np.mean(r64 * r64, axis=-1, keepdims=True))
    mag = (np.abs(O.bf16_to_f64(xb)) @ np.abs(O.bf16_to_f64(C.bits(wkv))).T).mean()
    abs_err = 4.0 * dim * 2.0 ** -24 * mag * rms
    assert np.all(np.abs(g64 - r64) <= ulp + abs_err), f"worst {np.max(np.abs(g64 - r64) - ulp - abs_err):.3e}"
    dist = _ulps_apart(got_lat, ref_lat)
    assert (dist > 0).mean() < 0.02, f"{(dist > 0).mean():.3%} of the latent differs"
    # weights_proj: the exactly rounded sum except within the f32 accumulation bound of a midpoint
    ref_w = O.weights_proj(xb, C.bits(wp))
    got_w = C.bits(w)
    a64, b64 = O.bf16_to_f64(xb).reshape(-1, dim), O.bf16_to_f64(C.bits(wp))
    exact = (a64 @ b64.T).reshape(got_w.shape)
    bound = dim * 2.0 ** -24 * (np.abs(a64) @ np.abs(b64).T).reshape(got_w.shape)
    err = np.abs(O.bf16_to_f64(got_w) - exact)
    assert np.all(err <= 2.0 ** -8 * np.abs(exact) + bound + 2.0 ** -133)
    diff = got_w != ref_w
    assert diff.mean() < 1e-2
    mid = 0.5 * (O.bf16_to_f64(got_w) + O.bf16_to_f64(ref_w))
    assert np.all((np.abs(exact - mid) <= bound + 2.0 ** -133)[diff] | (err[diff] <= bound[diff] + 2.0 ** -133))
    # the quantised latent: the oracle's quantiser of the kernel's own latent, bit for bit
    _, _, ref_q = O.fp4_quant_e4m3(got_lat)
    assert np.array_equal(C.bits(latq), ref_q)


def test_compress_feeds_the_key_publish_and_the_forward(X):
    """The producers' latent and head weights into indexer_forward_publish, against the oracle's
    publish and forward of the same latent and weights (bit-exact keys, scores within the
    tolerance, indices up to boundary swaps)."""
    wl = dataclasses.replace(WORKLOADS["prefill"], name="cp_e2e", B=1, S=512, ratio=4, H=64, dim=1024, topk=64)
    _, lat, _, w = _run(X, wl, with_q=False)
    d = C.dims_of(wl)
    table = C.gpu_table(wl.max_pos)
    cos, sin = C.oracle_table(wl.max_pos)
    cache = X.new_key_cache(wl.B, wl.T_cap)
    q = wl.q("cuda")
    ws = torch.empty(X.indexer_workspace_size(d, wl.B, wl.S, 0), dtype=torch.uint8, device="cuda")
    X.indexer_workspace_init(ws)
    top = torch.empty((wl.B, wl.S, wl.topk), dtype=torch.int32, device="cuda")
    sc = torch.empty((wl.B, wl.S, wl.T), dtype=torch.float32, device="cuda")
    X.indexer_forward_publish(d, lat, wl.wk("cuda"), wl.k_norm_w("cuda"), q, w, 0, table, cache, top, ws,
                              scores_out=sc)
    X.indexer_status(ws)
    ref_cache = C.oracle_cache(wl, cos, sin, latent=lat.cpu())
    assert np.array_equal(C.pages_to_rows(cache), ref_cache)
    ref_top, _, ref_sc = O.forward(C.bits(q), C.bits(w), ref_cache, cos, sin, 0, wl.ratio, wl.rope_dim, wl.topk,
                                   wl.offset)
    C.assert_scores_close(sc.cpu().numpy(), ref_sc)
    swaps = C.compare_topk(top.cpu().numpy().reshape(-1, wl.topk), ref_top.reshape(-1, wl.topk),
                           ref_sc.reshape(-1, wl.T), wl.offset)
    C.record_swaps("compress + forward", swaps, wl.S, int((top >= 0).sum()))
