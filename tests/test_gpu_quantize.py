"""GPU parity of ISQ (qmm_quantize) and qmm_dequantize: packed bytes and
dequantized fp32 weights must be bit-identical to the CPU oracle."""
import numpy as np
import pytest
import torch

import oracle
import ggml_block_quantized_linear_b300 as q
from ggml_block_quantized_linear_b300 import inputs
from qmm_testutil import DEV, to_dev_u8

pytestmark = pytest.mark.gpu
FMTS = [q.QMM_Q8_0, q.QMM_Q4_K]


def gpu_quantize(fmt, w_cpu):
    return q.qmm_quantize(fmt, w_cpu.to(DEV)).cpu().numpy()


def oracle_quantize(fmt, w_cpu):
    if w_cpu.dtype == torch.bfloat16:
        return oracle.quantize(fmt, inputs.bf16_bits(w_cpu))
    return oracle.quantize(fmt, w_cpu.numpy())


def assert_same_bytes(got, want, fmt):
    if not np.array_equal(got, want):
        diff = np.argwhere(got.reshape(-1) != want.reshape(-1))
        blk = oracle.BLOCK[fmt][1]
        i = int(diff[0][0])
        raise AssertionError("%d differing bytes; first at byte %d (block %d, offset %d): %d vs %d"
                             % (diff.size, i, i // blk, i % blk, got.reshape(-1)[i], want.reshape(-1)[i]))


@pytest.mark.parametrize("fmt", FMTS)
def test_tiny_fp32_linear_round_trip(fmt):
    # 256 x 512 fp32 weights ~ N(0, 0.02): quantize -> dequantize
    w = inputs.weights(256, 512, inputs.seed_for(1), fp32=True)
    got = gpu_quantize(fmt, w)
    want = oracle_quantize(fmt, w)
    assert_same_bytes(got, want, fmt)
    deq = q.qmm_dequantize(fmt, to_dev_u8(want), 256, 512).cpu().numpy()
    assert np.array_equal(deq.view(np.uint32), oracle.dequantize(fmt, want, 256, 512).view(np.uint32))


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("shape", inputs.DECODE_SHAPES)
def test_decode_shapes_bit_exact(fmt, shape):
    n, k = shape
    w = inputs.weights(n, k, inputs.seed_for(2 if fmt == q.QMM_Q8_0 else 3,
                                              inputs.DECODE_SHAPES.index(shape)))
    got = gpu_quantize(fmt, w)
    want = oracle_quantize(fmt, w)
    assert_same_bytes(got, want, fmt)
    deq = q.qmm_dequantize(fmt, to_dev_u8(want), n, k).cpu().numpy()
    ref = oracle.dequantize(fmt, want, n, k)
    assert np.array_equal(deq.view(np.uint32), ref.view(np.uint32))


def edge_cases():
    rng = np.random.default_rng(7)
    cases = {}
    cases["one_row"] = torch.from_numpy(rng.normal(0, 1, (1, 256)).astype(np.float32))
    cases["ragged_rows"] = torch.from_numpy(rng.normal(0, 0.02, (37, 768)).astype(np.float32))
    cases["zeros"] = torch.zeros((3, 512))
    cases["signed_zeros"] = -torch.zeros((2, 512))
    cases["tiny_subnormal_scales"] = torch.from_numpy(
        (rng.normal(0, 1, (8, 512)) * 1e-6).astype(np.float32))
    cases["mixed_magnitudes"] = torch.from_numpy(
        (rng.normal(0, 1, (8, 512)) * np.exp2(rng.integers(-30, 10, (8, 512)))).astype(np.float32))
    cases["all_negative"] = -torch.from_numpy(np.abs(rng.normal(0, 1, (4, 512))).astype(np.float32)) - 0.5
    cases["all_positive"] = torch.from_numpy(np.abs(rng.normal(0, 1, (4, 512))).astype(np.float32)) + 0.5
    cases["constant"] = torch.full((2, 512), 0.3)
    ties = np.zeros((4, 512), dtype=np.float32)  # values on half-steps of a power-of-two grid
    ties[:, :] = ((np.arange(512) % 64) - 31.5) * 2.0 ** -7
    ties[:, ::32] = 127 * 2.0 ** -7
    cases["ties"] = torch.from_numpy(ties)
    cases["large"] = torch.from_numpy(rng.normal(0, 1000, (4, 512)).astype(np.float32))
    # one float32 ulp either side of the half-steps: the reciprocal shortcut
    # of the quantizer must hand these to the exact division
    near = ties.copy()
    near[0] = np.nextafter(near[0], np.float32(np.inf))
    near[1] = np.nextafter(near[1], np.float32(-np.inf))
    near[2] = np.nextafter(np.nextafter(near[2], np.float32(np.inf)), np.float32(np.inf))
    near[:, ::32] = 127 * 2.0 ** -7
    cases["near_ties"] = torch.from_numpy(near.astype(np.float32))
    q4 = np.zeros((4, 512), dtype=np.float32)  # Q4_K grid: min 0, 15 steps of 2^-6
    q4[:, :] = ((np.arange(512) % 32) / 2.0) * 2.0 ** -6
    q4[1] = np.nextafter(q4[1], np.float32(np.inf))
    q4[2] = np.nextafter(q4[2], np.float32(-np.inf))
    cases["q4_half_steps"] = torch.from_numpy(q4)
    cases["q8_near_ties_scaled"] = torch.from_numpy(q8_near_ties_scaled(rng))
    cases["q4_near_ties_scaled"] = torch.from_numpy(q4_near_ties_scaled(rng))
    return cases


def _nudge(v, steps):
    """v moved by `steps` float32 ulps (elementwise, signed)."""
    v = v.astype(np.float32).copy()
    for s in range(int(np.abs(steps).max())):
        up = steps > s
        dn = -steps > s
        v[up] = np.nextafter(v[up], np.float32(np.inf))
        v[dn] = np.nextafter(v[dn], np.float32(-np.inf))
    return v


def q8_near_ties_scaled(rng, rows=16, cols=512):
    """Q8_0 blocks whose scale is a known binary16 value D (amax = 127 D, so
    amax / 127 = D exactly) and whose other weights lie a few float32 ulps
    from the half-steps (k + 1/2) D: quotients just inside and outside the
    tie guard of the reciprocal shortcut, with D not a power of two."""
    nb = rows * cols // 32
    D = np.ldexp(1.0 + rng.integers(0, 1024, nb) / 1024.0, rng.integers(-10, 4, nb)).astype(np.float32)
    k = rng.integers(-127, 127, (nb, 32)).astype(np.float32)
    x = _nudge((k + 0.5) * D[:, None], rng.integers(-12, 13, (nb, 32)))
    x[:, 0] = 127.0 * D
    return x.reshape(rows, cols)


def q4_near_ties_scaled(rng, rows=16, cols=512):
    """Q4_K superblocks with non-negative weights (so the min terms vanish),
    a known superblock scale D (sub-block 0 spans 15 * 63 D) and sub-block
    scale codes c_j (sub-block j spans 15 c_j D), so S_j = c_j D exactly;
    the other weights lie a few float32 ulps from (k + 1/2) S_j."""
    ns = rows * cols // 256
    D = np.ldexp(1.0 + rng.integers(0, 32, ns) / 32.0, rng.integers(-12, 2, ns)).astype(np.float32)
    c = rng.integers(1, 64, (ns, 8)).astype(np.float32)
    c[:, 0] = 63.0
    S = c * D[:, None]
    k = rng.integers(0, 15, (ns, 8, 32)).astype(np.float32)
    x = _nudge((k + 0.5) * S[:, :, None], rng.integers(-12, 13, (ns, 8, 32)))
    x[:, :, 0] = 15.0 * S
    x[:, :, 1] = 0.0
    return x.reshape(rows, cols)


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("name", sorted(edge_cases().keys()))
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_edge_cases_bit_exact(fmt, name, dtype):
    w = edge_cases()[name]
    if dtype == "bf16":
        w = w.to(torch.bfloat16)
    got = gpu_quantize(fmt, w.contiguous())
    want = oracle_quantize(fmt, w.contiguous())
    assert_same_bytes(got, want, fmt)
    rows, cols = w.shape
    deq = q.qmm_dequantize(fmt, to_dev_u8(want), rows, cols).cpu().numpy()
    assert np.array_equal(deq.view(np.uint32), oracle.dequantize(fmt, want, rows, cols).view(np.uint32))


@pytest.mark.parametrize("fmt", FMTS)
def test_empty_and_determinism(fmt):
    e = torch.empty((0, 256), dtype=torch.bfloat16, device=DEV)
    assert q.qmm_quantize(fmt, e).numel() == 0
    w = inputs.weights(300, 1024, 99).to(DEV)
    a = q.qmm_quantize(fmt, w)
    b = q.qmm_quantize(fmt, w)
    assert torch.equal(a, b)
    assert q.qmm_device_error_take() == 0
