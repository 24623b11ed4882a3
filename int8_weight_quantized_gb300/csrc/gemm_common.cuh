// gemm_common.cuh -- pieces of the tcgen05 GEMM kernel (gemm.cu) kept apart from its
// main loop: output types of the dequant epilogue, the bounded teardown wait, the wait
// limit.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ck_device.cuh"

namespace ck {
namespace gemm {

constexpr uint64_t DEFAULT_TIMEOUT_NS = 2000000000ull;  // 2 s per wait
constexpr uint32_t OUT_ROW_BYTES = 64;                  // a TMA store box is 32 rows x 64 bytes
constexpr uint32_t OUT_BUF_BYTES = 32 * OUT_ROW_BYTES;

// Bounded wait used during teardown only (never raises the abort flag again).
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, unsigned int* err,
                                           uint64_t timeout_ns)
{
    if (mbar_try_wait(bar, parity))
        return;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity))
            return;
        if ((i & 255u) == 0 && globaltimer_ns() - t0 > timeout_ns) {
            atomicOr(err, kErrWaitDrain);
            return;
        }
    }
}

// Output element types of the epilogue (the pages' int8_linear(..., out_dtype)).
enum : int { kOutBf16 = 0, kOutF16 = 1, kOutF32 = 2 };

template <int OUT>
struct OutType {
    static constexpr int BYTES = OUT == kOutF32 ? 4 : 2;
    static constexpr int BOX_COLS = (int)OUT_ROW_BYTES / BYTES;  // 32 (16-bit types) or 16 (fp32)
    static constexpr int PER_CHUNK = 16 / BYTES;                   // values per 16-byte chunk
};

// 16 bytes of output-type values -> fp32 (exact).
template <int OUT>
__device__ __forceinline__ void unpack_out(const uint4& r, float (&v)[OutType<OUT>::PER_CHUNK])
{
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
    if (OUT == kOutF32) {
#pragma unroll
        for (int i = 0; i < 4; ++i)
            v[i] = __uint_as_float(w[i]);
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            if (OUT == kOutF16) {
                const __half2 h = *reinterpret_cast<const __half2*>(&w[i]);
                v[2 * i] = __low2float(h);
                v[2 * i + 1] = __high2float(h);
            } else {
                const __nv_bfloat162 h = *reinterpret_cast<const __nv_bfloat162*>(&w[i]);
                v[2 * i] = __low2float(h);
                v[2 * i + 1] = __high2float(h);
            }
        }
    }
}

// Round two fp32 values to the output type and pack them (lower column first).
template <int OUT>
__device__ __forceinline__ uint32_t pack2(float lo, float hi)
{
    if (OUT == kOutF16) {
        __half2 v = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&v);
    } else {
        __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&v);
    }
}


}  // namespace gemm
}  // namespace ck
