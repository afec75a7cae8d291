"""Run one hot-path call on its configured shape a few times, for a profiler.

    python -m weight_streaming_warp_gb300.profile_case gemv_q8_0
    python -m weight_streaming_warp_gb300.profile_case quantize_gemv_q8_0
    python -m weight_streaming_warp_gb300.profile_case gemv_bf16 [M K]
    python -m weight_streaming_warp_gb300.profile_case gemm_bf16 [N]
    python -m weight_streaming_warp_gb300.profile_case dequant_kv [depth]
    python -m weight_streaming_warp_gb300.profile_case moe [T]
    python -m weight_streaming_warp_gb300.profile_case quantize [n block]
    python -m weight_streaming_warp_gb300.profile_case attn_decode [depth group]

Weights rotate over copies that together exceed the 129 MB L2, so every profiled
launch streams its weights from HBM; the device holds at most a few GB.  Inputs are
random (values do not change the work of these kernels).
"""
import sys

import torch

import weight_streaming_warp_gb300 as wsw


def main(argv):
    what = argv[0] if argv else "gemv_q8_0"
    dev = "cuda"
    g = torch.Generator(device=dev)
    g.manual_seed(0)
    launches = 6
    if what == "gemv_q8_0":
        M, K, nc = 14336, 4096, 4
        Wq = [torch.randint(-127, 128, (M, K), dtype=torch.int8, device=dev, generator=g) for _ in range(nc)]
        Wd = [(torch.rand((M, K // 32), device=dev, generator=g) * 1e-3).half() for _ in range(nc)]
        xq, xd = wsw.quantize_q8(torch.randn(K, device=dev, generator=g), 32)
        for i in range(launches):
            wsw.gemv_q8_0(Wq[i % nc], Wd[i % nc], xq, xd)
    elif what == "quantize_gemv_q8_0":
        M, K, nc = 14336, 4096, 4
        Wq = [torch.randint(-127, 128, (M, K), dtype=torch.int8, device=dev, generator=g) for _ in range(nc)]
        Wd = [(torch.rand((M, K // 32), device=dev, generator=g) * 1e-3).half() for _ in range(nc)]
        x = torch.randn((launches, K), device=dev, generator=g)
        xq = torch.empty(K, dtype=torch.int8, device=dev)
        xd = torch.empty(K // 32, dtype=torch.float16, device=dev)
        for i in range(launches):
            wsw.quantize_gemv_q8_0(Wq[i % nc], Wd[i % nc], x[i], x_out=(xq, xd))
    elif what == "gemv_bf16":
        M, K = (int(argv[1]), int(argv[2])) if len(argv) > 2 else (5120, 17408)
        nc = max(2, (512 << 20) // (M * K * 2) + 1)
        W = [torch.randn((M, K), device=dev, generator=g).to(torch.bfloat16) for _ in range(nc)]
        x = torch.randn(K, device=dev, generator=g)
        for i in range(launches):
            wsw.gemv_bf16(W[i % nc], x)
    elif what == "gemm_bf16":
        N = int(argv[1]) if len(argv) > 1 else 512
        M, K, nc = 2560, 10240, 4
        W = [torch.randn((M, K), device=dev, generator=g).mul_(0.02).to(torch.bfloat16) for _ in range(nc)]
        X = torch.randn((N, K), device=dev, generator=g).to(torch.bfloat16)
        for i in range(launches):
            wsw.gemm_bf16(W[i % nc], X)
    elif what == "dequant_kv":
        D = int(argv[1]) if len(argv) > 1 else 65536
        nc = 4
        q = [torch.randint(-127, 128, (D, 4, 128), dtype=torch.int8, device=dev, generator=g) for _ in range(nc)]
        d = [torch.rand((D, 4, 4), device=dev, generator=g).half() for _ in range(nc)]
        for i in range(launches):
            wsw.dequant_q8_0_kv(q[i % nc], d[i % nc])
    elif what == "moe":
        from weight_streaming_warp_gb300 import synthetic as syn
        T = int(argv[1]) if len(argv) > 1 else 16
        E, Mo, K = 128, 1536, 2048
        Wq = torch.randint(-127, 128, (E, Mo, K), dtype=torch.int8, device=dev, generator=g)
        Wd = (torch.rand((E, Mo, K // 32), device=dev, generator=g) * 1e-3).half()
        ids = syn.routing(0, "profile%d" % T, T, E, 8).to(dev)
        xq = torch.randint(-127, 128, (T * 8, K), dtype=torch.int8, device=dev, generator=g)
        xd = torch.rand((T * 8, K // 32), device=dev, generator=g).half()
        for _ in range(launches):
            wsw.moe_gemv_q8_0(Wq, Wd, xq, xd, ids)
    elif what == "attn_decode":
        D = int(argv[1]) if len(argv) > 1 else 32768
        G = int(argv[2]) if len(argv) > 2 else 1
        nc = 3  # 3 x 67 MB of K and V at depth 32768
        K = [torch.randn((4, D, 128), device=dev, generator=g).half() for _ in range(nc)]
        V = [torch.randn((4, D, 128), device=dev, generator=g).half() for _ in range(nc)]
        q = torch.randn((4, G, 128), device=dev, generator=g)
        for i in range(launches):
            wsw.attn_decode_f16(q, K[i % nc], V[i % nc])
    elif what == "quantize":
        n = int(argv[1]) if len(argv) > 1 else 4096
        block = int(argv[2]) if len(argv) > 2 else 32
        X = torch.randn((64, n), device=dev, generator=g)
        for i in range(launches):
            wsw.quantize_q8(X[i], block)
    else:
        raise SystemExit("unknown case %r" % what)
    torch.cuda.synchronize()
    print("done", what)


if __name__ == "__main__":
    main(sys.argv[1:])
