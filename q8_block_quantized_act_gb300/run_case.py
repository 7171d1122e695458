"""Launch one kernel of libq8act on one shape, for profilers (no timing, no checking).

    python -m q8_block_quantized_act_gb300.run_case gemv --m 1 --n 64448 --k 4096 --reps 3
    python -m q8_block_quantized_act_gb300.run_case gemm --m 512 --n 4096 --k 4096 --reps 2

Kernels: quantize (q8_1), quantize_mmq, quantize_q8_0, gemv, gemm (fused quantize),
gemm_preq, gemm_repacked (fused quantize, load-time repacked weights), repack, dequant,
gemv_q4_0, dequant_q4_0, and the K-quant passes gemv_q6_k / gemv_q4_k / gemv_q5_k and
dequant_q6_k / dequant_q4_k / dequant_q5_k (on seeded random superblocks).
Inputs are the seeded synthetic ones of q8_block_quantized_act_gb300.inputs;
one warm-up launch precedes the `--reps` launches.
"""
from __future__ import annotations

import argparse


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("kernel", choices=("quantize", "quantize_mmq", "quantize_q8_0", "gemv", "gemm",
                                       "gemm_preq", "gemm_repacked", "repack", "dequant", "gemv_q4_0",
                                       "dequant_q4_0", "gemv_q6_k", "gemv_q4_k", "gemv_q5_k",
                                       "dequant_q6_k", "dequant_q4_k", "dequant_q5_k"))
    ap.add_argument("--m", type=int, default=1)
    ap.add_argument("--n", type=int, default=4096)
    ap.add_argument("--k", type=int, default=4096)
    ap.add_argument("--reps", type=int, default=1)
    a = ap.parse_args(argv)

    import torch
    import q8_block_quantized_act_gb300 as q8
    from q8_block_quantized_act_gb300 import build as q8build
    from q8_block_quantized_act_gb300 import inputs

    q8build.build()
    dev = torch.device("cuda")
    m, n, k = a.m, a.n, a.k
    x = torch.from_numpy(inputs.activations_f32(m, k)).to(dev)
    need_w = a.kernel in ("gemv", "gemm", "gemm_preq", "gemm_repacked", "repack", "dequant")
    w = q8.quantize_q8_0(torch.from_numpy(inputs.weights_f32(n, k)).to(dev)) if need_w else None
    w32 = torch.from_numpy(inputs.weights_f32(n, k)).to(dev) if a.kernel == "quantize_q8_0" else None
    w4 = (q8.quantize_q4_0(torch.from_numpy(inputs.weights_f32(n, k)).to(dev))
          if a.kernel in ("gemv_q4_0", "dequant_q4_0") else None)
    xq, xd = q8.quantize_q8_1(x)
    xqh, xdt = q8.quantize_q8_1_mmq(x)
    kq = a.kernel.split("_", 1)[1] if a.kernel.endswith("_k") else None   # "q6_k", "q4_k", "q5_k"
    wk = torch.from_numpy(inputs.kquant_superblocks(kq, n, k)).to(dev) if kq else None
    ws = q8.gemm_workspace(m, k, dev) if a.kernel in ("gemm", "gemm_repacked") else None
    wq16, wdt = q8.repack_q8_0(w, n, k) if a.kernel in ("gemm_repacked", "repack") else (None, None)
    torch.cuda.synchronize()

    def once():
        if a.kernel == "quantize":
            q8.quantize_q8_1(x)
        elif a.kernel == "quantize_mmq":
            q8.quantize_q8_1_mmq(x)
        elif a.kernel == "quantize_q8_0":
            q8.quantize_q8_0(w32)
        elif a.kernel == "gemv":
            q8.gemv_q8_0(w, xq, xd, n)
        elif a.kernel == "gemm":
            q8.gemm_q8_0(w, x, n, ws=ws)
        elif a.kernel == "gemm_preq":
            q8.gemm_q8_0_preq(w, xqh, xdt, n)
        elif a.kernel == "gemm_repacked":
            q8.gemm_q8_0_repacked(wq16, wdt, x, ws=ws)
        elif a.kernel == "repack":
            q8.check(q8.q8act_repack_q8_0(w, wq16, wdt, n, k))
        elif a.kernel == "gemv_q4_0":
            q8.gemv_q4_0(w4, xq, xd, n)
        elif a.kernel == "dequant_q4_0":
            q8.dequant_q4_0_f16(w4, n, k)
        elif kq and a.kernel.startswith("gemv"):
            q8.gemv_kq(kq, wk, xq, xd, n)
        elif kq:
            q8.dequant_kq_f16(kq, wk, n, k)
        else:
            q8.dequant_q8_0_f16(w, n, k)

    for _ in range(1 + a.reps):
        once()
    torch.cuda.synchronize()
    q8.device_status()
    print(f"ran {a.kernel} m={m} n={n} k={k} x{1 + a.reps}")


if __name__ == "__main__":
    main()
