"""Run one operation of the library once (after one warm-up call) on seeded
synthetic inputs, for profilers such as Nsight Compute.

    python -m bit_quantized_tensor_gb300.profile_case OP [--m M] [--n N] [--k K]

OP is one of s8, s4, f16 (M x N x K GEMMs), w4a16 (M x N x K with group 128),
w4a4_quant (M x K activations with rank-32 projection) or w4a4_gemm
(M x N x K, rank 32, bias).  Sizes default to 2048 each.  Prints one line
with the call's device time from CUDA events (a number taken under a
profiler is not a benchmark figure).
"""
import argparse
import sys

import numpy as np


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawTextHelpFormatter)
    ap.add_argument("op", choices=["s8", "s4", "f16", "w4a16", "w4a4_quant", "w4a4_gemm"])
    ap.add_argument("--m", type=int, default=2048)
    ap.add_argument("--n", type=int, default=2048)
    ap.add_argument("--k", type=int, default=2048)
    a = ap.parse_args(argv)

    import torch

    import bit_quantized_tensor_gb300 as qg
    from bit_quantized_tensor_gb300 import inputs

    if not torch.cuda.is_available():
        sys.exit("profile_case needs a CUDA device")
    dev = torch.device("cuda:0")
    qg.lib()
    M, N, K = a.m, a.n, a.k

    def t(x):
        return torch.from_numpy(np.ascontiguousarray(x)).to(dev)

    if a.op == "s8":
        A, B = t(inputs.s8_uniform(M, K, 1000)), t(inputs.s8_uniform(N, K, 2000))
        run = lambda: qg.qgemm_s8(A, B)  # noqa: E731
    elif a.op == "s4":
        A, B = t(inputs.s4_packed_uniform(M, K, 1001)), t(inputs.s4_packed_uniform(N, K, 2001))
        run = lambda: qg.qgemm_s4(A, B, K)  # noqa: E731
    elif a.op == "f16":
        A, B = t(inputs.f16_normal(M, K, 1002)), t(inputs.f16_normal(N, K, 2002))
        run = lambda: qg.gemm_f16(A, B)  # noqa: E731
    elif a.op == "w4a16":
        X = t(inputs.f16_normal(M, K, 1003))
        Wq = t(inputs.s4_packed_uniform(N, K, 2003))
        S = t(inputs.f16_uniform(N, K // 128, 0.005, 0.02, 3003))
        run = lambda: qg.w4a16_gemm(X, Wq, S)  # noqa: E731
    elif a.op == "w4a4_quant":
        X = t(inputs.f32_normal(M, K, 1004))
        Ut = t(inputs.f16_normal(K, 32, 3004, sigma=0.02).T)
        run = lambda: qg.w4a4_quantize(X, Ut)  # noqa: E731
    else:
        X = t(inputs.f32_normal(M, K, 1004))
        W = t(inputs.f32_normal(N, K, 2004))
        Ut = t(inputs.f16_normal(K, 32, 3004, sigma=0.02).T)
        Vt = t(inputs.f16_normal(32, N, 3005, sigma=0.02).T)
        b = t(inputs.f16_normal(1, N, 3006, sigma=0.1)[0])
        qx, sx, xu = qg.w4a4_quantize(X, Ut)
        qw, sw, _ = qg.w4a4_quantize(W)
        del X, W
        run = lambda: qg.w4a4_gemm(qx, sx, qw, sw, K, XU=xu, Vt=Vt, bias=b)  # noqa: E731

    run()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    run()
    e1.record()
    torch.cuda.synchronize()
    assert qg.device_status() == qg.QG_OK
    print(f"{a.op} M={M} N={N} K={K}: {e0.elapsed_time(e1) * 1e3:.1f} us (one call)")


if __name__ == "__main__":
    main()
