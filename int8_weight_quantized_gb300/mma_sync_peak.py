"""Measure the dense rate of the warp-level tensor-core instructions (mma.sync) on this GPU.

    python -m int8_weight_quantized_gb300.mma_sync_peak

sm_103a has no int8 kind of the tcgen05 instructions, so its only int8 x int8 -> int32 matrix
instruction is the warp-level mma.sync.m16n8k32.s32.s8.s8.s32 inherited from earlier GPUs.  This
tool times it (and the bf16 mma.sync.m16n8k16 for comparison) with register-resident operands:
every warp issues chains of independent MMAs, enough warps on every SM to keep the pipe busy,
nothing read from memory.  The figures are the GPU's dense int8 / bf16 rates through that
instruction family, the denominator an int8 GEMM on mma.sync could at best reach.  The kernel
source is compiled here with nvcc for sm_103a (it is not part of the library).
"""
import argparse
import ctypes
import os
import subprocess
import tempfile

from . import build as _build

SRC = r"""
#include <cstdint>
#include <cuda_runtime.h>

// CHAINS independent accumulators per warp, each fed by the same register operands.
template <int CHAINS>
__global__ void __launch_bounds__(256) mma_s8(int iters, int* out)
{
    uint32_t a0 = threadIdx.x * 0x01010101u, a1 = a0 + 1, a2 = a0 + 2, a3 = a0 + 3;
    uint32_t b0 = blockIdx.x * 0x01010101u, b1 = b0 + 5;
    int c[CHAINS][4];
#pragma unroll
    for (int j = 0; j < CHAINS; ++j)
        c[j][0] = c[j][1] = c[j][2] = c[j][3] = 0;
    for (int i = 0; i < iters; ++i) {
#pragma unroll
        for (int j = 0; j < CHAINS; ++j)
            asm volatile("mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
                         "{%8, %9}, {%0, %1, %2, %3};"
                         : "+r"(c[j][0]), "+r"(c[j][1]), "+r"(c[j][2]), "+r"(c[j][3])
                         : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    }
    int s = 0;
#pragma unroll
    for (int j = 0; j < CHAINS; ++j)
        s += c[j][0] ^ c[j][1] ^ c[j][2] ^ c[j][3];
    if (s == 0x12345678)  // never true in practice; keeps the MMAs live
        out[0] = s;
}

template <int CHAINS>
__global__ void __launch_bounds__(256) mma_bf16(int iters, float* out)
{
    uint32_t a0 = 0x3F803F80u + threadIdx.x, a1 = a0 + 1, a2 = a0 + 2, a3 = a0 + 3;
    uint32_t b0 = 0x3F803F80u + blockIdx.x, b1 = b0 + 5;
    float c[CHAINS][4];
#pragma unroll
    for (int j = 0; j < CHAINS; ++j)
        c[j][0] = c[j][1] = c[j][2] = c[j][3] = 0.0f;
    for (int i = 0; i < iters; ++i) {
#pragma unroll
        for (int j = 0; j < CHAINS; ++j)
            asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
                         "{%8, %9}, {%0, %1, %2, %3};"
                         : "+f"(c[j][0]), "+f"(c[j][1]), "+f"(c[j][2]), "+f"(c[j][3])
                         : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    }
    float s = 0.0f;
#pragma unroll
    for (int j = 0; j < CHAINS; ++j)
        s += c[j][0] + c[j][1] + c[j][2] + c[j][3];
    if (s == 1.2345f)
        out[0] = s;
}

// Returns the average time in ms of `reps` launches (after one untimed launch), or a
// negative CUDA error code.
extern "C" double run(int kind, int blocks, int iters, int reps)
{
    void* out = nullptr;
    if (cudaMalloc(&out, 16) != cudaSuccess)
        return -1.0;
    cudaEvent_t e0, e1;
    cudaEventCreate(&e0);
    cudaEventCreate(&e1);
    auto launch = [&] {
        if (kind == 0)
            mma_s8<8><<<blocks, 256>>>(iters, static_cast<int*>(out));
        else
            mma_bf16<8><<<blocks, 256>>>(iters, static_cast<float*>(out));
    };
    launch();
    cudaEventRecord(e0);
    for (int r = 0; r < reps; ++r)
        launch();
    cudaEventRecord(e1);
    cudaError_t err = cudaEventSynchronize(e1);
    float ms = 0.0f;
    cudaEventElapsedTime(&ms, e0, e1);
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    cudaFree(out);
    if (err != cudaSuccess)
        return -(double)err;
    return ms / reps;
}
"""


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--iters", type=int, default=512)
    ap.add_argument("--reps", type=int, default=5)
    args = ap.parse_args(argv)
    import torch  # the device's SM count; the measurement itself is the CUDA source above

    sms = torch.cuda.get_device_properties(0).multi_processor_count
    with tempfile.TemporaryDirectory() as d:
        src = os.path.join(d, "mma_sync_peak.cu")
        lib = os.path.join(d, "mma_sync_peak.so")
        with open(src, "w") as f:
            f.write(SRC)
        subprocess.run([_build.nvcc(), *_build.ARCH, "-O3", "-shared", "-Xcompiler", "-fPIC", "-o", lib, src],
                       check=True)
        L = ctypes.CDLL(lib)
        L.run.restype = ctypes.c_double
        L.run.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int]
        for kind, name, flops_per_mma in ((0, "int8 mma.sync.m16n8k32 (s32 accumulate)", 2 * 16 * 8 * 32),
                                          (1, "bf16 mma.sync.m16n8k16 (f32 accumulate)", 2 * 16 * 8 * 16)):
            best = None
            for per_sm in (2, 4, 8):
                blocks = per_sm * sms
                ms = L.run(kind, blocks, args.iters, args.reps)
                if ms < 0:
                    raise RuntimeError("CUDA error %d" % int(-ms))
                rate = blocks * 8 * 8 * args.iters * flops_per_mma / (ms * 1e-3) / 1e12  # 8 warps, 8 chains
                print("%s: %d blocks of 256 threads, %.3f ms, %.1f T(FL)OP/s" % (name, blocks, ms, rate), flush=True)
                best = rate if best is None else max(best, rate)
            print("%s: best %.1f T(FL)OP/s" % (name, best), flush=True)


if __name__ == "__main__":
    main()
