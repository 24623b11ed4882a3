// ck_internal.h -- host-side interface between the C ABI (api.cu) and the kernels
// (quantize.cu, gemm.cu).  Not installed; the public contract is include/ck_int8.h.
#pragma once

#include <cstddef>
#include <cstdint>
#include <mutex>
#include <string>
#include <utility>
#include <vector>

#include <cuda_runtime.h>

namespace ck {

// Launch `kernel` with programmatic stream serialization, so its launch and prologue
// overlap the tail of the previous kernel on the stream (the kernel itself calls
// griddep_wait() before reading or writing global memory).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args&&... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// One tensor-core GEMM problem: A [M,K] and B [N,K] are bf16 tensors whose values are
// integers in [-127, 127] (the int8 codes, widened); the kernel forms the exact
// integer products and either dequantizes them (y != nullptr) or writes the raw int32
// accumulators (acc != nullptr).
struct GemmProblem {
    const void* a = nullptr;
    const void* b = nullptr;
    int64_t M = 0, N = 0, K = 0;
    const float* x_scale = nullptr;
    const float* w_scale = nullptr;
    const void* bias = nullptr;  // bf16 [N] or nullptr
    const void* residual = nullptr;  // [M,N] of the output type or nullptr (may alias y)
    int scalar_scales = 0;
    void* y = nullptr;           // [M,N] of the output type
    int out_dtype = 0;           // 0 bf16, 1 fp16, 2 fp32
    void* tail = nullptr;        // gemm_tail_bytes(M, N) bytes of workspace (K-split tail)
    bool mixed = false;          // a = 16-bit activations, fp32 sum over all of K, no x_scale
    int32_t* acc = nullptr;      // int32 [M,N]
};

struct DeviceInfo {
    int device = -1;
    int major = 0, minor = 0;
    int sm_count = 0;
};

// Query (once per device) and return the current device's properties.
cudaError_t current_device(DeviceInfo* info);

// Identifier of the CUDA context current on this host thread, unique for the life of
// the process (the driver's context id).  With no context current yet, the current
// device's primary context is made current first.
cudaError_t current_context_id(unsigned long long* id);

// A value that belongs to a CUDA context (a device address of one of the library's
// variables, a kernel attribute set on it), made once per context by make(&value) while
// that context is current.  A device reset creates a new context with a new id, so the
// value is made again there instead of reusing what belonged to the destroyed one.
template <typename T>
class ContextCache {
public:
    template <typename Make>
    cudaError_t get(T* out, Make make)
    {
        unsigned long long id = 0;
        cudaError_t e = current_context_id(&id);
        if (e != cudaSuccess)
            return e;
        std::lock_guard<std::mutex> lock(mu_);
        for (const auto& kv : entries_)
            if (kv.first == id) {
                *out = kv.second;
                return cudaSuccess;
            }
        T v{};
        if ((e = make(&v)) != cudaSuccess)
            return e;
        entries_.emplace_back(id, v);
        *out = v;
        return cudaSuccess;
    }

private:
    std::mutex mu_;
    std::vector<std::pair<unsigned long long, T>> entries_;
};

// Kernel launchers.  Each returns cudaSuccess or the launch error; `why` gets a
// description of a failure that is not a CUDA error.
// The GEMM's K-split tail keeps, per CTA slice of a split unit, 128 x 256 int32 partial
// sums and 8 arrival slots of 16 bytes in the caller's workspace; at most
// gemm_tail_ctas(M, N) CTA slices, a bound that needs no device query.
constexpr int kTailMaxSplit = 8;
constexpr int64_t kTailMaxCtas = 152;
constexpr size_t kTailCtaBytes = (size_t)128 * 256 * 4;
constexpr size_t kTailSlotBytesPerCta = (size_t)8 * 16;
inline int64_t gemm_tail_ctas(int64_t M, int64_t N)
{
    const int64_t slices = ((M + 127) / 128) * ((N + 31) / 32) * kTailMaxSplit;
    return slices < kTailMaxCtas ? slices : kTailMaxCtas;
}
inline size_t gemm_tail_bytes(int64_t M, int64_t N)
{
    return (size_t)gemm_tail_ctas(M, N) * (kTailCtaBytes + kTailSlotBytesPerCta);
}

// The GEMM launch configuration for an M x N x K problem: CTA pairs or single CTAs, the
// tile width (a multiple of 32 up to 256), how many units can be resident at once, and
// the K-split of the last partial wave (split = 1: none).
struct GemmPlan {
    bool pair = false;
    int bn = 0;
    int64_t resident = 0;
    int64_t units = 0;       // units of the whole problem
    int64_t full_units = 0;  // units computed whole; the rest are split
    int split = 1;
};
cudaError_t plan_gemm(int64_t M, int64_t N, int64_t K, bool mixed, const DeviceInfo& dev, GemmPlan* plan);
cudaError_t launch_gemm(const GemmProblem& p, const DeviceInfo& dev, cudaStream_t s, std::string* why);
cudaError_t launch_quantize_rows(const void* x, int64_t M, int64_t K, bool rotate, int8_t* q8, void* q16,
                                 float* x_scale, const DeviceInfo& dev, cudaStream_t s);
// Tensorwise quantize in two launches: per-block maxima into `partials`
// (tensorwise_partials() floats), then the quantize pass, which first reduces them.
int tensorwise_partials(const DeviceInfo& dev);
cudaError_t launch_quantize_tensorwise(const void* x, int64_t M, int64_t K, int8_t* q8, void* q16,
                                       float* x_scale, float* partials, const DeviceInfo& dev, cudaStream_t s);
// The same two launches with the number of partial maxima chosen by the caller
// (`partials` holds at least nparts floats).
cudaError_t launch_quantize_tensorwise_parts(const void* x, int64_t M, int64_t K, int8_t* q8, void* q16,
                                             float* x_scale, float* partials, int nparts, const DeviceInfo& dev,
                                             cudaStream_t s);
// The layer's preparation in one launch: quantize the activation into bf16 codes (and
// its scales) and widen the int8 weight w8 (w_n values) into w16.  Per-row / ConvRot:
// the row kernel takes a share of the widening.  Tensorwise: a single kernel whose
// blocks exchange their maxima through `scratch` (prep_tensorwise_scratch_bytes(max_blocks)
// bytes of workspace; its content on entry does not matter).
cudaError_t launch_prep_rows(const void* x, int64_t M, int64_t K, bool rotate, void* q16, float* x_scale,
                             const int8_t* w8, int64_t w_n, void* w16, const DeviceInfo& dev, cudaStream_t s);
size_t prep_tensorwise_scratch_bytes(int max_blocks);
cudaError_t launch_prep_tensorwise(const void* x, int64_t M, int64_t K, void* q16, float* x_scale, void* scratch,
                                   int max_blocks, const int8_t* w8, int64_t w_n, void* w16, const DeviceInfo& dev,
                                   cudaStream_t s);
// 16-bit-activation ConvRot operand: a16 = bf16(x @ H) ([M,K], K % 128 == 0), plus the
// int8 -> bf16 weight widening, in one launch.
cudaError_t launch_rotate_bf16(const void* x, int64_t M, int64_t K, void* a16, const int8_t* w8, int64_t w_n,
                               void* w16, const DeviceInfo& dev, cudaStream_t s);
// Two int8 -> bf16 widenings in one launch.
cudaError_t launch_widen2(const int8_t* a8, int64_t a_n, void* a16, const int8_t* b8, int64_t b_n, void* b16,
                          const DeviceInfo& dev, cudaStream_t s);
// ConvRot weight preparation: W fp32 [N,K] -> int8 codes of W @ H^T and fp32 row scales.
cudaError_t launch_convrot_weight(const float* W, int64_t N, int64_t K, int8_t* w, float* w_scale,
                                  const DeviceInfo& dev, cudaStream_t s);
// Device address of the library's error word on the current device.
cudaError_t device_error_ptr(unsigned int** ptr);
// int8 -> bf16 widening of n values (n % 16 == 0).
cudaError_t launch_widen_int8(const int8_t* src, void* dst, int64_t n, const DeviceInfo& dev, cudaStream_t s);

// Device error word (bits in ck_device.cuh).
cudaError_t read_device_error(unsigned int* value, bool clear);
cudaError_t launch_wait_selftest(uint64_t timeout_ns, cudaStream_t s);

// Diagnostics: one line per unique problem shape when CK_LOG=1 (log_enabled()).
bool log_enabled();
void log_shape(const char* what, int64_t M, int64_t N, int64_t K, int mode, const std::string& engine);
// "<bn>-wide tiles on CTA pairs / single CTAs, K split s ways in the last wave" for the
// GEMM an M x N x K launch would run (for the CK_LOG lines).
std::string describe_gemm_plan(int64_t M, int64_t N, int64_t K, bool mixed, bool split_allowed,
                               const DeviceInfo& dev);

}  // namespace ck
