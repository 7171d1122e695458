"""Stream order under programmatic dependent launches.

Most of the library's kernels may become resident while the previous kernel of the stream
still runs and wait for it before touching memory; the second kernel of a fused call streams
weights before that wait, relying on its quantizer having started only after everything before
it completed.  Here a kernel that rewrites a weight buffer and the library calls that read it
follow each other on one stream with no host synchronization, the buffer's contents changing
every iteration; every result must equal, bit for bit, the same call made on its own between
device synchronizations."""
import pytest
import torch

import q8_block_quantized_act_gb300 as q8
from q8_block_quantized_act_gb300 import inputs
from gpu_util import device_ok, ensure_built

pytestmark = pytest.mark.gpu


def test_q8_0_calls_see_the_previous_kernels_writes():
    ensure_built()
    n, k, mg, mv = 4096, 4096, 64, 8
    dev = torch.device("cuda")
    w32 = [torch.from_numpy(inputs.weights_f32(n, k, seed=s)).to(dev) for s in (11, 12, 13)]
    x1 = torch.from_numpy(inputs.activations_f32(1, k)).to(dev)
    xv = torch.from_numpy(inputs.activations_f32(mv, k, seed=5)).to(dev)
    xg = torch.from_numpy(inputs.activations_f32(mg, k, seed=6)).to(dev)

    xq, xd = q8.quantize_q8_1(xv)

    def calls(wq):
        return (lambda: q8.gemv_q8_0_f32(wq, x1, n),    # fused: streams weights before its wait
                lambda: q8.gemm_q8_0(wq, xg, n),        # fused GEMM
                lambda: q8.dequant_q8_0_f16(wq, n, k),
                lambda: q8.gemv_q8_0(wq, xq, xd, n))    # the tensor-core GEMV (m = 8)

    refs = []
    for w in w32:
        wq = q8.quantize_q8_0(w)
        outs = []
        for c in calls(wq):
            torch.cuda.synchronize()
            outs.append(c())
        torch.cuda.synchronize()
        refs.append(outs)

    wq = torch.empty((n, k // 32 * 34), dtype=torch.uint8, device=dev)
    chained = []
    for it in range(6):
        q8.check(q8.q8act_quantize_q8_0(w32[it % 3], wq, n, k))   # rewrites the weights
        chained.append([c() for c in calls(wq)])
    torch.cuda.synchronize()
    device_ok()
    for it, outs in enumerate(chained):
        for j, (a, b) in enumerate(zip(outs, refs[it % 3])):
            assert torch.equal(a, b), (it, j)


def test_k_quant_calls_see_the_previous_kernels_writes():
    ensure_built()
    n, k = 4096, 4096
    dev = torch.device("cuda")
    x = torch.from_numpy(inputs.activations_f32(8, k)).to(dev)
    xq, xd = q8.quantize_q8_1(x)
    for fmt in ("q6_k", "q4_k", "q5_k"):
        src = [torch.from_numpy(inputs.kquant_superblocks(fmt, n, k, seed=s)).to(dev) for s in (21, 22)]

        def calls(wk):
            return (lambda: q8.gemv_kq(fmt, wk, xq[:1], xd[:1], n),   # dp4a kernel
                    lambda: q8.gemv_kq(fmt, wk, xq, xd, n),           # tensor-core kernel (m = 8)
                    lambda: q8.dequant_kq_f16(fmt, wk, n, k))

        refs = []
        for s in src:
            outs = []
            for c in calls(s):
                torch.cuda.synchronize()
                outs.append(c())
            torch.cuda.synchronize()
            refs.append(outs)
        wk = torch.empty_like(src[0])
        chained = []
        for it in range(4):
            torch.bitwise_or(src[it % 2], 0, out=wk)   # an elementwise kernel rewrites the superblocks
            chained.append([c() for c in calls(wk)])
        torch.cuda.synchronize()
        device_ok()
        for it, outs in enumerate(chained):
            for j, (a, b) in enumerate(zip(outs, refs[it % 2])):
                assert torch.equal(a, b), (fmt, it, j)
