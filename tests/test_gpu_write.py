"""GPU cache write vs the oracle: stored code and scale bytes bit-exact.

Every catalogue format (both sides in one launch), head_dim 64/128/256,
fp32 and bf16 activations, K/V read through fused-QKV strides, a ragged
token count with skipped (-1) slots, padded block strides, and a slot past
the pool that must be flagged instead of written."""
import numpy as np
import pytest
import torch

import oracle
from quantized_paged_kv_reshape_gb300 import ops
from kvq_cases import ALL_FORMATS, bf16_round, fp8_scales

pytestmark = pytest.mark.gpu


def run_write(fmt, hd, in_dtype, nkv=2, bs=16, num_blocks=7, ntok=45, seed=0, pad=32,
              bad_slot=False, row_extra=8, shift=0):
    """Fused QKV rows of (nq + 2 nkv) * hd + row_extra elements; K and V start
    `shift` elements after their heads' natural offsets in the row."""
    assert 0 <= shift <= row_extra
    rng = np.random.default_rng(seed)
    nq = 2 * nkv
    row = (nq + 2 * nkv) * hd + row_extra   # fused QKV row, stride != nkv*hd
    fused = rng.standard_normal((ntok, row)).astype(np.float32)
    fused[:, rng.choice(row, 6, replace=False)] *= 10.0      # outlier channels
    fused[3, :] = 0.0                                         # an all-zero token
    if in_dtype == "bf16":
        fused = bf16_round(fused)
    slots = rng.permutation(num_blocks * bs)[:ntok].astype(np.int64)
    slots[rng.choice(ntok, 5, replace=False)] = -1
    if bad_slot:
        slots[7] = num_blocks * bs + 3
    koff, voff = nq * hd + shift, (nq + nkv) * hd + shift
    kview = fused[:, koff:koff + nkv * hd].reshape(ntok, nkv, hd)
    vview = fused[:, voff:voff + nkv * hd].reshape(ntok, nkv, hd)
    kside, vside = oracle.kv_pair(fmt)
    ks, vs = fp8_scales(kview, vview)
    kst = (oracle.block_bytes(kside, bs, nkv, hd) + 15) // 16 * 16 + pad
    vst = (oracle.block_bytes(vside, bs, nkv, hd) + 15) // 16 * 16 + pad
    kc = np.zeros(num_blocks * kst, np.uint8)
    vc = np.zeros(num_blocks * vst, np.uint8)
    ok_slots = np.where(slots < num_blocks * bs, slots, -1)
    oracle.cache_write(kside, kview, kc, ok_slots, nkv, hd, bs, kst, scale=ks)
    oracle.cache_write(vside, vview, vc, ok_slots, nkv, hd, bs, vst, scale=vs)

    dev = "cuda"
    tdt = torch.bfloat16 if in_dtype == "bf16" else torch.float32
    fused_d = torch.from_numpy(fused).to(dev).to(tdt)
    kpool = torch.zeros((num_blocks, kst), dtype=torch.uint8, device=dev)
    vpool = torch.zeros((num_blocks, vst), dtype=torch.uint8, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    ops.cache_write(fused_d[:, koff:], fused_d[:, voff:], kpool, vpool,
                    torch.from_numpy(slots).to(dev), fmt, nkv, hd, bs, key_stride=row,
                    value_stride=row, k_scale=ks, v_scale=vs, error_flag=err)
    torch.cuda.synchronize()
    return kc, vc, kpool.cpu().numpy().reshape(-1), vpool.cpu().numpy().reshape(-1), int(err.item())


@pytest.mark.parametrize("in_dtype", ["f32", "bf16"])
@pytest.mark.parametrize("hd", [64, 128, 256])
@pytest.mark.parametrize("fmt", ALL_FORMATS)
def test_write_bit_exact(fmt, hd, in_dtype):
    kc, vc, kg, vg, err = run_write(fmt, hd, in_dtype, seed=hd)
    assert err == 0
    assert np.array_equal(kc, kg), f"K bytes differ at {np.flatnonzero(kc != kg)[:8]}"
    assert np.array_equal(vc, vg), f"V bytes differ at {np.flatnonzero(vc != vg)[:8]}"


@pytest.mark.parametrize("row_extra,shift", [(1, 0), (3, 1)])
@pytest.mark.parametrize("in_dtype", ["f32", "bf16"])
@pytest.mark.parametrize("hd", [64, 128, 256])
@pytest.mark.parametrize("fmt", ALL_FORMATS)
def test_write_unaligned_strides(fmt, hd, in_dtype, row_extra, shift):
    """Key/value rows whose per-token stride (an odd element count) or start
    (one element past a 16-byte boundary) breaks the lanes' vector alignment:
    the library must take the per-element loads and store the same bytes."""
    kc, vc, kg, vg, err = run_write(fmt, hd, in_dtype, seed=hd + 7, row_extra=row_extra,
                                    shift=shift)
    assert err == 0
    assert np.array_equal(kc, kg), f"K bytes differ at {np.flatnonzero(kc != kg)[:8]}"
    assert np.array_equal(vc, vg), f"V bytes differ at {np.flatnonzero(vc != vg)[:8]}"


@pytest.mark.parametrize("fmt", ["turbo4", "bf16k_turbo3v", "fp8k_turbo2v", "turbo8"])
def test_write_flags_slot_past_pool(fmt):
    kc, vc, kg, vg, err = run_write(fmt, 128, "bf16", bad_slot=True)
    assert err & 1
    assert np.array_equal(kc, kg) and np.array_equal(vc, vg)


@pytest.mark.parametrize("nkv,bs", [(1, 8), (3, 16), (16, 32)])
def test_write_shapes(nkv, bs):
    for fmt in ("turbo3", "turbo2", "fp8k_turbo4v"):
        kc, vc, kg, vg, err = run_write(fmt, 128, "bf16", nkv=nkv, bs=bs, num_blocks=9, ntok=60)
        assert np.array_equal(kc, kg) and np.array_equal(vc, vg)


def test_write_empty_is_noop():
    dev = "cuda"
    kpool = torch.zeros((2, 4096), dtype=torch.uint8, device=dev)
    x = torch.zeros((1, 256), dtype=torch.bfloat16, device=dev)
    ops.cache_write(x, x, kpool, kpool, torch.zeros(0, dtype=torch.int64, device=dev),
                    "turbo4", 2, 128, 16)
    torch.cuda.synchronize()
    assert not kpool.any()


def _near_threshold_rows(side, hd, rng):
    """Rows whose quantizer inputs y sit within a few ulps of a decision
    boundary times the group scale: element 0 of every group fixes the scale
    (amax = largest level x s, s an E4M3 value), the others are a boundary x s
    nudged by -3..3 ulps.  Boundaries: the Lloyd-Max midpoint thresholds, or
    the E2M1 midpoints for nvfp4."""
    if side == "nvfp4":
        bounds, top = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], np.float32), 6.0
    else:
        bits = oracle.formats.CODE_BITS[side]
        _, lv32, thr = oracle.codebook(bits)
        bounds, top = thr.astype(np.float32), float(lv32[-1])
    scales = oracle.e4m3_decode(np.arange(0x08, 0x7E, dtype=np.uint8)).astype(np.float32)
    n_groups = 512
    y = np.zeros((n_groups, 16), np.float32)
    for g in range(n_groups):
        s = scales[rng.integers(len(scales))]
        y[g, 0] = np.float32(top) * s
        b = bounds[rng.integers(len(bounds), size=15)]
        v = (b * s).astype(np.float32)
        steps = rng.integers(-3, 4, size=15)
        for i in range(15):
            for _ in range(abs(steps[i])):
                v[i] = np.nextafter(v[i], np.float32(np.inf if steps[i] > 0 else -np.inf))
        y[g, 1:] = v * rng.choice(np.array([-1, 1], np.float32), 15)
    y = y.reshape(-1, hd)
    # Rotated sides quantize WHT(x): feed x = WHT(y) (fp32, self-inverse up to
    # rounding), so the kernel's rotated values land within a few ulps of y.
    return y if side == "nvfp4" else oracle.fwht_f32(y)


@pytest.mark.parametrize("fmt", ["turbo4", "turbo3", "turbo2", "nvfp4"])
@pytest.mark.parametrize("hd", [64, 128, 256])
def test_write_near_decision_boundaries(fmt, hd):
    """Codes of values a few ulps from a threshold: the kernel's quotient and
    code search must round exactly like the oracle's fp32 division."""
    rng = np.random.default_rng(hd)
    nkv, bs = 2, 16
    x = _near_threshold_rows(fmt, hd, rng).astype(np.float32)
    ntok = x.shape[0] // nkv
    x = x[: ntok * nkv].reshape(ntok, nkv, hd)
    num_blocks = -(-ntok // bs)
    slots = np.arange(ntok, dtype=np.int64)
    st = (oracle.block_bytes(fmt, bs, nkv, hd) + 15) // 16 * 16
    kc = np.zeros(num_blocks * st, np.uint8)
    oracle.cache_write(fmt, x, kc, slots, nkv, hd, bs, st)
    xd = torch.from_numpy(x).cuda()
    kpool = torch.zeros((num_blocks, st), dtype=torch.uint8, device="cuda")
    vpool = torch.zeros((num_blocks, st), dtype=torch.uint8, device="cuda")
    ops.cache_write(xd.view(ntok, -1), xd.view(ntok, -1), kpool, vpool,
                    torch.from_numpy(slots).cuda(), fmt, nkv, hd, bs)
    torch.cuda.synchronize()
    got = kpool.cpu().numpy().reshape(-1)
    assert np.array_equal(got, kc), f"{int((got != kc).sum())} bytes differ"


def test_write_graph_replay():
    """The write captures into a CUDA graph, as a serving step replays it:
    after the input rows and the slots are refilled, each replay stores the
    oracle's bytes for the new rows (an odd token count: the last warp's
    second half-warp row has no token)."""
    fmt, hd, nkv, bs, nb, ntok = "turbo4k_turbo3v", 128, 2, 16, 7, 31
    kside, vside = oracle.kv_pair(fmt)
    kst = (oracle.block_bytes(kside, bs, nkv, hd) + 15) // 16 * 16
    vst = (oracle.block_bytes(vside, bs, nkv, hd) + 15) // 16 * 16
    dev = "cuda"
    k_d = torch.zeros((ntok, nkv * hd), device=dev)
    v_d = torch.zeros((ntok, nkv * hd), device=dev)
    s_d = torch.full((ntok,), -1, dtype=torch.int64, device=dev)
    kpool = torch.zeros((nb, kst), dtype=torch.uint8, device=dev)
    vpool = torch.zeros((nb, vst), dtype=torch.uint8, device=dev)

    def call():
        ops.cache_write(k_d, v_d, kpool, vpool, s_d, fmt, nkv, hd, bs)

    call()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    torch.cuda.synchronize()
    rng = np.random.default_rng(17)
    for _ in range(2):
        k = rng.standard_normal((ntok, nkv, hd)).astype(np.float32)
        v = rng.standard_normal((ntok, nkv, hd)).astype(np.float32)
        slots = rng.permutation(nb * bs)[:ntok].astype(np.int64)
        slots[rng.choice(ntok, 3, replace=False)] = -1
        k_d.copy_(torch.from_numpy(k.reshape(ntok, -1)))
        v_d.copy_(torch.from_numpy(v.reshape(ntok, -1)))
        s_d.copy_(torch.from_numpy(slots))
        kpool.zero_()
        vpool.zero_()
        g.replay()
        torch.cuda.synchronize()
        kc = np.zeros(nb * kst, np.uint8)
        vc = np.zeros(nb * vst, np.uint8)
        oracle.cache_write(kside, k, kc, slots, nkv, hd, bs, kst)
        oracle.cache_write(vside, v, vc, slots, nkv, hd, bs, vst)
        assert np.array_equal(kpool.cpu().numpy().reshape(-1), kc)
        assert np.array_equal(vpool.cpu().numpy().reshape(-1), vc)


def _write_pair(fmt, k, v, slots, nkv, hd, bs, num_blocks, ks=1.0, vs=1.0, in_dtype="f32"):
    """Oracle bytes and GPU bytes of one write of K rows k and V rows v."""
    kside, vside = oracle.kv_pair(fmt)
    kst = (oracle.block_bytes(kside, bs, nkv, hd) + 15) // 16 * 16
    vst = (oracle.block_bytes(vside, bs, nkv, hd) + 15) // 16 * 16
    kc = np.zeros(num_blocks * kst, np.uint8)
    vc = np.zeros(num_blocks * vst, np.uint8)
    oracle.cache_write(kside, k, kc, slots, nkv, hd, bs, kst, scale=ks)
    oracle.cache_write(vside, v, vc, slots, nkv, hd, bs, vst, scale=vs)
    tdt = torch.bfloat16 if in_dtype == "bf16" else torch.float32
    ntok = k.shape[0]
    kd = torch.from_numpy(k.reshape(ntok, -1)).cuda().to(tdt)
    vd = torch.from_numpy(v.reshape(ntok, -1)).cuda().to(tdt)
    kpool = torch.zeros((num_blocks, kst), dtype=torch.uint8, device="cuda")
    vpool = torch.zeros((num_blocks, vst), dtype=torch.uint8, device="cuda")
    ops.cache_write(kd, vd, kpool, vpool, torch.from_numpy(slots).cuda(), fmt, nkv, hd, bs,
                    k_scale=ks, v_scale=vs)
    torch.cuda.synchronize()
    return kc, vc, kpool.cpu().numpy().reshape(-1), vpool.cpu().numpy().reshape(-1)


@pytest.mark.parametrize("in_dtype", ["f32", "bf16"])
@pytest.mark.parametrize("hd", [64, 128, 256])
@pytest.mark.parametrize("fmt", ["turbo4", "turbo3", "turbo2", "nvfp4", "turbo8",
                                 "turbo4k_turbo3v", "bf16k_turbo2v"])
def test_write_extreme_magnitudes(fmt, hd, in_dtype):
    """Rows scaled so that group scales saturate at E4M3's 448 (the quotients
    then run far past the top level), land in E4M3's subnormal range or round
    to zero, all-zero rows, -0 elements and lone spikes: bytes equal the
    oracle's."""
    rng = np.random.default_rng(hd + (7 if in_dtype == "bf16" else 0))
    nkv, bs = 2, 16
    factors = np.array([3e5, 2e3, 1.0, 1e-3, 3e-5, 1e-7, 1e-30, 0.0], np.float32)
    ntok = 2 * len(factors)
    k = rng.standard_normal((ntok, nkv, hd)).astype(np.float32)
    v = rng.standard_normal((ntok, nkv, hd)).astype(np.float32)
    for t in range(ntok):
        k[t] *= factors[t % len(factors)]
        v[t] *= factors[(t + 3) % len(factors)]
    k[1, 0, :] = -0.0                                   # a row of -0
    v[2, 1, ::3] = -0.0                                 # -0 elements among values
    k[5, 1, :] = 0.0
    k[5, 1, 17] = -4e4                                  # a lone spike
    v[6, 0, :] = 1e-3
    v[6, 0, 40] = 9e3
    if in_dtype == "bf16":
        k, v = bf16_round(k), bf16_round(v)
    slots = rng.permutation(ntok).astype(np.int64)
    kc, vc, kg, vg = _write_pair(fmt, k, v, slots, nkv, hd, bs, 1, in_dtype=in_dtype)
    assert np.array_equal(kc, kg), f"K bytes differ at {np.flatnonzero(kc != kg)[:8]}"
    assert np.array_equal(vc, vg), f"V bytes differ at {np.flatnonzero(vc != vg)[:8]}"


@pytest.mark.parametrize("scales", [(1.0, 0.25), (3.0, 0.37), (2.0 ** -20, 2.0 ** 20)])
@pytest.mark.parametrize("hd", [64, 128, 256])
def test_write_fp8_scales(hd, scales):
    """FP8 codes of x / scale: powers of two (a product with the exact
    reciprocal) and other scales (a division) round like the oracle's fp32
    division, saturating at 448."""
    rng = np.random.default_rng(hd)
    nkv, bs, ntok = 3, 16, 21
    ks, vs = scales
    k = (rng.standard_normal((ntok, nkv, hd)) * 40 * ks).astype(np.float32)
    v = (rng.standard_normal((ntok, nkv, hd)) * 40 * vs).astype(np.float32)
    k[0, 0, :4] = [1e30, -1e30, -0.0, 0.0]
    slots = rng.permutation(2 * bs)[:ntok].astype(np.int64)
    kc, vc, kg, vg = _write_pair("fp8", k, v, slots, nkv, hd, bs, 2, ks=ks, vs=vs)
    assert np.array_equal(kc, kg), f"K bytes differ at {np.flatnonzero(kc != kg)[:8]}"
    assert np.array_equal(vc, vg), f"V bytes differ at {np.flatnonzero(vc != vg)[:8]}"
