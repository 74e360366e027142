"""GPU parity for the whole-model workload and for chained calls.

* The synthetic 8B-shape decoder (32 layers x 7 linears, weights generated on
  the GPU with the bench's seeds): for the first and the last layer, ISQ of
  every linear in both formats on the GPU is compared byte for byte with the
  oracle on a sample of rows, and the M = 1 decode output on those rows is
  compared element by element with the oracle's fp64 product.
* Chained calls, as a decode step issues them: ISQ output consumed by the next
  matmul, one matmul's output (cast to bf16) fed to the next, and a matmul
  whose output overwrites the previous matmul's input.  The decode kernels
  start early (programmatic dependent launch) and must still see the previous
  kernel's writes and not overwrite what it reads.  Run eagerly and as a CUDA
  graph; the graph replay must give the same bits.
"""
import numpy as np
import pytest
import torch

import oracle
import ggml_block_quantized_linear_b300 as q
from ggml_block_quantized_linear_b300 import inputs
from qmm_testutil import DEV, check_matmul

pytestmark = pytest.mark.gpu
FMTS = [q.QMM_Q8_0, q.QMM_Q4_K]


def sample_rows(n, count, seed):
    rng = np.random.default_rng(seed)
    s = set(rng.choice(n, size=min(count, n), replace=False).tolist())
    s.update([0, n - 1, 15, 16])
    return np.array(sorted(s), dtype=np.int64)


@pytest.mark.parametrize("layer", [0, inputs.MODEL_LAYERS - 1])
@pytest.mark.parametrize("li", range(len(inputs.MODEL_LINEARS)))
def test_model_layer_isq_and_decode(layer, li):
    name, n, k = inputs.MODEL_LINEARS[li]
    w = inputs.weights(n, k, inputs.model_weight_seed(layer, li), device=DEV)
    x = inputs.activations(1, k, inputs.model_activation_seed(layer, li), device=DEV)
    rows = sample_rows(n, 48, 100 * layer + li)
    wb = inputs.bf16_bits(w[torch.from_numpy(rows).to(DEV)])
    xb = inputs.bf16_bits(x)
    for fmt in FMTS:
        packed = q.qmm_quantize(fmt, w)
        y = q.qmm_matmul(fmt, packed, x, n)
        want = oracle.quantize(fmt, wb)
        got = packed[torch.from_numpy(rows).to(DEV)].cpu().numpy()
        assert np.array_equal(got, want), "%s layer %d fmt %d: packed bytes differ" % (name, layer, fmt)
        Y, A = oracle.matmul(fmt, want, xb, rows.size, k)
        check_matmul(y[:, torch.from_numpy(rows).to(DEV)], Y, A, "%s layer %d fmt %d" % (name, layer, fmt))
    assert q.qmm_device_error_take() == 0


def _chain(fmt, ws, x0, outs, packs):
    """ISQ of each weight, then the chain x -> W0 -> bf16 -> W1 -> ..."""
    x = x0
    for i, w in enumerate(ws):
        q.qmm_quantize(fmt, w, out=packs[i])
        q.qmm_matmul(fmt, packs[i], x, w.shape[0], out=outs[i])
        x = outs[i].to(torch.bfloat16)
    return outs


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("m", [1, 4, 16])
def test_chained_decode_eager_and_graph(fmt, m):
    # q (4096 x 4096) -> o (4096 x 4096) -> gate (14336 x 4096) -> down (4096 x 14336)
    shapes = [(4096, 4096), (4096, 4096), (14336, 4096), (4096, 14336)]
    ws = [inputs.weights(n, k, 700 + i, device=DEV) for i, (n, k) in enumerate(shapes)]
    x0 = inputs.activations(m, 4096, 701, device=DEV)
    packs = [torch.empty((n, q.qmm_packed_bytes(fmt, n, k) // n), dtype=torch.uint8, device=DEV)
             for n, k in shapes]
    outs = [torch.empty((m, n), dtype=torch.float32, device=DEV) for n, _ in shapes]
    _chain(fmt, ws, x0, outs, packs)
    torch.cuda.synchronize()
    eager = [o.clone() for o in outs]
    # every link against the oracle, with the bf16 input that link really saw
    xs = [x0] + [o.to(torch.bfloat16) for o in eager[:-1]]
    for i, (n, k) in enumerate(shapes):
        rows = sample_rows(n, 32, 10 * i + m)
        packed = oracle.quantize(fmt, inputs.bf16_bits(ws[i][torch.from_numpy(rows).to(DEV)]))
        Y, A = oracle.matmul(fmt, packed, inputs.bf16_bits(xs[i]), rows.size, k)
        check_matmul(eager[i][:, torch.from_numpy(rows).to(DEV)], Y, A, "link %d" % i)
    # the same chain captured once and replayed
    for o in outs:
        o.zero_()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            _chain(fmt, ws, x0, outs, packs)
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    for a, b in zip(eager, outs):
        assert torch.equal(a, b)
    assert q.qmm_device_error_take() == 0


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("m", [1, 16])
@pytest.mark.parametrize("n1", [4096, 1024])
def test_next_call_overwrites_previous_input(fmt, m, n1):
    # call A reads X from `buf`; call B, next in the stream, writes its output
    # into the same bytes.  B may start before A has finished, but it must not
    # write before A is complete.
    k1 = 4096  # n1 = 1024: the cluster split-K kernel reads X
    n2, k2 = 4096, 4096
    w1 = inputs.weights(n1, k1, 801, device=DEV)
    w2 = inputs.weights(n2, k2, 802, device=DEV)
    p1, p2 = q.qmm_quantize(fmt, w1), q.qmm_quantize(fmt, w2)
    xa = inputs.activations(m, k1, 803, device=DEV)
    xb = inputs.activations(m, k2, 804, device=DEV)
    buf = torch.empty(m * n2 * 4, dtype=torch.uint8, device=DEV)
    xa_view = buf[: m * k1 * 2].view(torch.bfloat16).view(m, k1)
    yb_view = buf.view(torch.float32).view(m, n2)
    ya_ref = q.qmm_matmul(fmt, p1, xa, n1)
    yb_ref = q.qmm_matmul(fmt, p2, xb, n2)
    for _ in range(3):
        xa_view.copy_(xa)
        ya = torch.empty((m, n1), dtype=torch.float32, device=DEV)
        q.qmm_matmul(fmt, p1, xa_view, n1, out=ya)
        q.qmm_matmul(fmt, p2, xb, n2, out=yb_view)
        torch.cuda.synchronize()
        assert torch.equal(ya, ya_ref)
        assert torch.equal(yb_view, yb_ref)
    assert q.qmm_device_error_take() == 0

