// api.cu -- the extern "C" boundary declared in include/ck_int8.h: argument checks,
// device check, workspace layout, and the launch sequence of each entry point.
// Every entry point validates before it enqueues anything and never synchronises the
// host (except the two diagnostics at the end).
#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <mutex>
#include <set>
#include <string>
#include <tuple>
#include <vector>

#include <cuda.h>
#include <cuda_runtime.h>

#include "ck_int8.h"
#include "ck_internal.h"

namespace ck {
namespace {

thread_local std::string g_last_error;

int fail(int status, const char* fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return status;
}

int cuda_fail(cudaError_t e, const char* where)
{
    return fail(CK_ERR_CUDA, "%s: %s (%s)", where, cudaGetErrorString(e), cudaGetErrorName(e));
}

bool aligned16(const void* p)
{
    return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

constexpr size_t kAlign = 256;
size_t align_up(size_t v)
{
    return (v + kAlign - 1) & ~(kAlign - 1);
}

constexpr int64_t kMaxDim = 0x7FFFFFFF;  // tensor-copy coordinates are 32-bit
constexpr int64_t kMaxK = 131072;        // 127*127*K must fit int32

// Checks shared by the GEMM entry points.  Returns CK_OK or a status with the message set.
int check_gemm_shape(int64_t M, int64_t N, int64_t K)
{
    if (M < 0 || N <= 0 || K <= 0)
        return fail(CK_ERR_INVALID_ARG, "M must be >= 0 and N, K >= 1 (got M=%lld N=%lld K=%lld)", (long long)M,
                    (long long)N, (long long)K);
    if (M > kMaxDim || N > kMaxDim)
        return fail(CK_ERR_INVALID_ARG, "M and N must each be < 2^31 (got M=%lld N=%lld)", (long long)M,
                    (long long)N);
    if (K % 16 != 0)
        return fail(CK_ERR_INVALID_ARG, "K must be a multiple of 16 (got %lld)", (long long)K);
    if (K > kMaxK)
        return fail(CK_ERR_INVALID_ARG, "K must be <= %lld so the int32 accumulator cannot overflow (got %lld)",
                    (long long)kMaxK, (long long)K);
    if (N % 8 != 0)
        return fail(CK_ERR_INVALID_ARG, "N must be a multiple of 8 (got %lld)", (long long)N);
    return CK_OK;
}

int check_device(DeviceInfo* dev)
{
    cudaError_t e = current_device(dev);
    if (e != cudaSuccess)
        return cuda_fail(e, "querying the current device");
    if (dev->major != 10 || dev->minor != 3)
        return fail(CK_ERR_UNSUPPORTED_DEVICE,
                    "this library is built for GB300 (compute capability 10.3); device %d is %d.%d", dev->device,
                    dev->major, dev->minor);
    return CK_OK;
}

#define CK_REQUIRE_PTR(p)                                                                       \
    do {                                                                                        \
        if ((p) == nullptr)                                                                     \
            return fail(CK_ERR_INVALID_ARG, "%s must not be NULL", #p);                         \
        if (!aligned16(p))                                                                      \
            return fail(CK_ERR_INVALID_ARG, "%s must be 16-byte aligned", #p);                  \
    } while (0)

constexpr int kMaxPartialsForLayout = 1024;  // most blocks that exchange tensorwise maxima

struct LinearWorkspace {
    void* a16;        // bf16 [M,K]: quantized activation as tensor-core operand
    void* b16;        // bf16 [N,K]: weight as tensor-core operand
    float* xs;        // fp32 [M] or [1]
    void* scratch;    // tensorwise: the blocks' maxima, exchanged within one launch
    void* tail;       // the GEMM's K-split tail: partial sums and arrival slots
};

// own_b16: the workspace holds the widened weight (ck_int8_linear); without it the caller
// passes the weight's codes (ck_int8_linear_codes).
size_t linear_ws_bytes(int64_t M, int64_t N, int64_t K, int mode, int nparts, bool own_b16 = true)
{
    return align_up((size_t)M * K * 2) + (own_b16 ? align_up((size_t)N * K * 2) : 0) +
           align_up(sizeof(float) * (size_t)(mode == CK_TENSORWISE ? 1 : (M > 0 ? M : 1))) +
           align_up(prep_tensorwise_scratch_bytes(nparts)) + align_up(gemm_tail_bytes(M, N));
}

LinearWorkspace carve_linear(void* ws, int64_t M, int64_t N, int64_t K, int mode, bool own_b16 = true)
{
    uint8_t* p = static_cast<uint8_t*>(ws);
    LinearWorkspace w;
    w.a16 = p;
    p += align_up((size_t)M * K * 2);
    w.b16 = own_b16 ? p : nullptr;
    if (own_b16)
        p += align_up((size_t)N * K * 2);
    w.xs = reinterpret_cast<float*>(p);
    p += align_up(sizeof(float) * (size_t)(mode == CK_TENSORWISE ? 1 : (M > 0 ? M : 1)));
    w.scratch = p;
    p += align_up(prep_tensorwise_scratch_bytes(kMaxPartialsForLayout));
    w.tail = p;
    return w;
}

size_t gemm_ws_bytes(int64_t M, int64_t N, int64_t K)
{
    return align_up((size_t)M * K * 2) + align_up((size_t)N * K * 2) + align_up(gemm_tail_bytes(M, N));
}

const int kMaxPartials = kMaxPartialsForLayout;

// ---- launch profiling: events around each kernel launch while enabled -------------
enum ProfKind { kProfQuantize = 0, kProfWiden = 1, kProfGemm = 2, kProfKinds = 3 };
struct ProfRec {
    int kind;
    int launches;
    cudaEvent_t a, b;
};
thread_local bool g_prof_on = false;
thread_local bool g_prof_events = false;
thread_local int64_t g_prof_counts[kProfKinds] = {};
thread_local std::vector<ProfRec> g_prof_recs;
thread_local std::vector<cudaEvent_t> g_prof_pool;

cudaEvent_t prof_event()
{
    if (!g_prof_pool.empty()) {
        cudaEvent_t e = g_prof_pool.back();
        g_prof_pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess)
        return nullptr;
    return e;
}

// Brackets the launches made in its lifetime with two events on `s` when profiling is on.
struct ProfScope {
    bool active = false;
    ProfRec r{};
    cudaStream_t s;
    ProfScope(int kind, int launches, cudaStream_t st) : s(st)
    {
        if (!g_prof_on)
            return;
        g_prof_counts[kind] += launches;
        if (!g_prof_events)
            return;
        r.kind = kind;
        r.launches = launches;
        r.a = prof_event();
        r.b = prof_event();
        active = r.a && r.b && cudaEventRecord(r.a, s) == cudaSuccess;
    }
    ~ProfScope()
    {
        if (active && cudaEventRecord(r.b, s) == cudaSuccess)
            g_prof_recs.push_back(r);
    }
};

}  // namespace

cudaError_t current_device(DeviceInfo* info)
{
    static DeviceInfo cache[64];
    static std::mutex mu;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    std::lock_guard<std::mutex> lock(mu);
    if (dev >= 0 && dev < 64 && cache[dev].device == dev) {
        *info = cache[dev];
        return cudaSuccess;
    }
    DeviceInfo d;
    d.device = dev;
    if ((e = cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
        return e;
    if (dev >= 0 && dev < 64)
        cache[dev] = d;
    *info = d;
    return cudaSuccess;
}

cudaError_t current_context_id(unsigned long long* id)
{
    using GetCurrentFn = CUresult (*)(CUcontext*);
    using GetIdFn = CUresult (*)(CUcontext, unsigned long long*);
    static GetCurrentFn get_current = nullptr;
    static GetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<GetCurrentFn>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<GetIdFn>(p);
    });
    if (get_current == nullptr || get_id == nullptr)
        return cudaErrorNotSupported;
    CUcontext ctx = nullptr;
    if (get_current(&ctx) != CUDA_SUCCESS)
        return cudaErrorDeviceUninitialized;
    if (ctx == nullptr) {
        // nothing current yet: the runtime would create the device's primary context on
        // its first real call; do that now so the id is the one later calls will see
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e == cudaSuccess)
            e = cudaSetDevice(dev);
        if (e != cudaSuccess)
            return e;
        if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr)
            return cudaErrorDeviceUninitialized;
    }
    return get_id(ctx, id) == CUDA_SUCCESS ? cudaSuccess : cudaErrorDeviceUninitialized;
}

bool log_enabled()
{
    static const bool on = [] {
        const char* v = std::getenv("CK_LOG");
        return v && v[0] == '1';
    }();
    return on;
}

void log_shape(const char* what, int64_t M, int64_t N, int64_t K, int mode, const std::string& engine)
{
    if (!log_enabled())
        return;
    static std::mutex mu;
    static std::set<std::tuple<std::string, int64_t, int64_t, int64_t, int>> seen;
    std::lock_guard<std::mutex> lock(mu);
    if (seen.insert(std::make_tuple(std::string(what), M, N, K, mode)).second)
        fprintf(stderr, "[ck] %s M=%lld N=%lld K=%lld mode=%d engine=%s\n", what, (long long)M, (long long)N,
                (long long)K, mode, engine.c_str());
}

}  // namespace ck

using namespace ck;

extern "C" {

const char* ck_last_error(void)
{
    return g_last_error.c_str();
}

int ck_quantize_int8_rowwise(const void* x, int64_t M, int64_t K, int rotate, int8_t* q, float* x_scale,
                             void* stream)
{
    if (M < 0 || K <= 0)
        return fail(CK_ERR_INVALID_ARG, "M must be >= 0 and K >= 1 (got M=%lld K=%lld)", (long long)M, (long long)K);
    if (K % 16 != 0)
        return fail(CK_ERR_INVALID_ARG, "K must be a multiple of 16 (got %lld)", (long long)K);
    if (rotate != 0 && rotate != 1)
        return fail(CK_ERR_INVALID_ARG, "rotate must be 0 or 1 (got %d)", rotate);
    if (rotate && K % 128 != 0)
        return fail(CK_ERR_INVALID_ARG, "the ConvRot rotation needs K % 128 == 0 (got %lld)", (long long)K);
    if (M == 0)
        return CK_OK;  // nothing to do; empty buffers may be NULL
    CK_REQUIRE_PTR(x);
    CK_REQUIRE_PTR(q);
    CK_REQUIRE_PTR(x_scale);
    DeviceInfo dev;
    int st = check_device(&dev);
    if (st != CK_OK)
        return st;
    log_shape("quantize_rowwise", M, 0, K, rotate ? CK_CONVROT : CK_PER_ROW, "rows (32-256 threads per row)");
    cudaError_t e;
    {
        ProfScope ps(kProfQuantize, 1, static_cast<cudaStream_t>(stream));
        e = launch_quantize_rows(x, M, K, rotate != 0, q, nullptr, x_scale, dev, static_cast<cudaStream_t>(stream));
    }
    return e == cudaSuccess ? CK_OK : cuda_fail(e, "ck_quantize_int8_rowwise launch");
}

size_t ck_quantize_tensorwise_workspace_size(void)
{
    return sizeof(float) * kMaxPartials;
}

int ck_quantize_int8_tensorwise(const void* x, int64_t M, int64_t K, int8_t* q, float* x_scale, void* workspace,
                                size_t workspace_bytes, void* stream)
{
    if (M < 0 || K <= 0)
        return fail(CK_ERR_INVALID_ARG, "M must be >= 0 and K >= 1 (got M=%lld K=%lld)", (long long)M, (long long)K);
    if (K % 16 != 0)
        return fail(CK_ERR_INVALID_ARG, "K must be a multiple of 16 (got %lld)", (long long)K);
    if (M == 0)
        return CK_OK;  // no maximum to take and nothing to quantize
    CK_REQUIRE_PTR(x);
    CK_REQUIRE_PTR(q);
    CK_REQUIRE_PTR(x_scale);
    CK_REQUIRE_PTR(workspace);
    if (workspace_bytes < ck_quantize_tensorwise_workspace_size())
        return fail(CK_ERR_INVALID_ARG, "workspace too small: %zu bytes given, %zu needed", workspace_bytes,
                    ck_quantize_tensorwise_workspace_size());
    DeviceInfo dev;
    int st = check_device(&dev);
    if (st != CK_OK)
        return st;
    log_shape("quantize_tensorwise", M, 0, K, CK_TENSORWISE, "block maxima, then quantize (2 launches)");
    cudaError_t e;
    {
        ProfScope ps(kProfQuantize, 2, static_cast<cudaStream_t>(stream));
        e = launch_quantize_tensorwise(x, M, K, q, nullptr, x_scale, static_cast<float*>(workspace), dev,
                                       static_cast<cudaStream_t>(stream));
    }
    return e == cudaSuccess ? CK_OK : cuda_fail(e, "ck_quantize_int8_tensorwise launch");
}

size_t ck_int8_linear_workspace_size(int64_t M, int64_t N, int64_t K, int mode)
{
    if (M < 0 || N < 0 || K < 0)
        return 0;
    return linear_ws_bytes(M, N, K, mode, kMaxPartials);
}

int ck_int8_linear_workspace_views(int64_t M, int64_t N, int64_t K, int mode, size_t* codes_offset,
                                   size_t* x_scale_offset)
{
    if (mode != CK_TENSORWISE && mode != CK_PER_ROW && mode != CK_CONVROT)
        return fail(CK_ERR_INVALID_ARG, "mode must be 0 (tensorwise), 1 (per-row) or 2 (ConvRot), got %d", mode);
    if (M < 0 || N < 0 || K < 0)
        return fail(CK_ERR_INVALID_ARG, "M, N and K must be >= 0");
    if (codes_offset == nullptr || x_scale_offset == nullptr)
        return fail(CK_ERR_INVALID_ARG, "codes_offset and x_scale_offset must not be NULL");
    uint8_t* const base = reinterpret_cast<uint8_t*>(kAlign);  // any aligned base: only differences are used
    const LinearWorkspace w = carve_linear(base, M, N, K, mode);
    *codes_offset = (size_t)(static_cast<uint8_t*>(w.a16) - base);
    *x_scale_offset = (size_t)(reinterpret_cast<uint8_t*>(w.xs) - base);
    return CK_OK;
}

// Whether work enqueued on `s` is being captured into a CUDA graph.  A captured launch
// replays with the arguments it was captured with, so the per-launch tags that the
// single-launch tensorwise preparation (block maxima exchanged in tagged slots) and the
// GEMM's K-split tail (tagged arrival counters) take from the host would repeat on every
// replay, and a replay could read the previous replay's maxima or miscount its arrivals.
// Under capture the layer therefore uses forms without tags: the two-launch tensorwise
// quantize (per-block maxima, then a pass that reduces them), a separate weight widening,
// and no K-split.
static bool stream_capturing(cudaStream_t s)
{
    cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
    return cudaStreamIsCapturing(s, &st) == cudaSuccess && st != cudaStreamCaptureStatusNone;
}

static bool valid_out_dtype(int t)
{
    return t == CK_OUT_BF16 || t == CK_OUT_F16 || t == CK_OUT_F32;
}

// The layer: w8 (int8 codes, widened by the preparation launch) or w_codes (the weight's
// bf16 codes, prepared once by ck_int8_weight_codes).
// The layer, from the int8 weight (own_b16: the preparation launch widens it into the
// workspace) or from the caller's prepared bf16 weight codes (w_codes).
static int linear_impl(const char* name, bool own_b16, const void* x, const int8_t* w8, const void* w_codes,
                       const float* w_scale, const void* bias, const void* residual, void* y, int64_t M, int64_t N,
                       int64_t K, int mode, int out_dtype, void* workspace, size_t workspace_bytes, void* stream)
{
    if (mode != CK_TENSORWISE && mode != CK_PER_ROW && mode != CK_CONVROT)
        return fail(CK_ERR_INVALID_ARG, "mode must be 0 (tensorwise), 1 (per-row) or 2 (ConvRot), got %d", mode);
    if (!valid_out_dtype(out_dtype))
        return fail(CK_ERR_INVALID_ARG, "out_dtype must be 0 (bf16), 1 (fp16) or 2 (fp32), got %d", out_dtype);
    int st = check_gemm_shape(M, N, K);
    if (st != CK_OK)
        return st;
    if (mode == CK_CONVROT && K % 128 != 0)
        return fail(CK_ERR_INVALID_ARG, "ConvRot needs K % 128 == 0 (got %lld)", (long long)K);
    if (M == 0)
        return CK_OK;  // empty batch: x and y may be NULL
    CK_REQUIRE_PTR(x);
    if (own_b16)
        CK_REQUIRE_PTR(w8);
    else
        CK_REQUIRE_PTR(w_codes);
    CK_REQUIRE_PTR(w_scale);
    CK_REQUIRE_PTR(y);
    CK_REQUIRE_PTR(workspace);
    if (bias != nullptr && !aligned16(bias))
        return fail(CK_ERR_INVALID_ARG, "bias must be 16-byte aligned");
    if (residual != nullptr && !aligned16(residual))
        return fail(CK_ERR_INVALID_ARG, "residual must be 16-byte aligned");
    const size_t need = linear_ws_bytes(M, N, K, mode, kMaxPartials, own_b16);
    if (workspace_bytes < need)
        return fail(CK_ERR_INVALID_ARG, "workspace too small: %zu bytes given, %zu needed", workspace_bytes, need);
    DeviceInfo dev;
    if ((st = check_device(&dev)) != CK_OK)
        return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    LinearWorkspace ws = carve_linear(workspace, M, N, K, mode, own_b16);
    const void* b16 = own_b16 ? ws.b16 : w_codes;
    const bool graph = stream_capturing(s);
    if (log_enabled())
        log_shape(name, M, N, K, mode,
                  std::string(mode == CK_TENSORWISE && graph ? "quantize (2 launches)" : "preparation (1 launch)") +
                      (own_b16 ? " with the weight widening" : ", weight codes given") +
                      " + tcgen05 bf16-exact GEMM, " + describe_gemm_plan(M, N, K, false, !graph, dev));
    cudaError_t e;
    if (mode == CK_TENSORWISE && graph) {
        // captured: per-block maxima, a quantize pass that reduces them, the widening apart
        ProfScope ps(kProfQuantize, 2, s);
        e = launch_quantize_tensorwise(x, M, K, nullptr, ws.a16, ws.xs, static_cast<float*>(ws.scratch), dev, s);
        if (e == cudaSuccess && own_b16)
            e = launch_widen_int8(w8, ws.b16, N * K, dev, s);
    } else {
        // one launch: quantize the activation into bf16 codes (and widen the weight)
        ProfScope ps(kProfQuantize, 1, s);
        if (mode == CK_TENSORWISE)
            e = launch_prep_tensorwise(x, M, K, ws.a16, ws.xs, ws.scratch, kMaxPartialsForLayout,
                                       own_b16 ? w8 : nullptr, N * K, ws.b16, dev, s);
        else
            e = launch_prep_rows(x, M, K, mode == CK_CONVROT, ws.a16, ws.xs, own_b16 ? w8 : nullptr, N * K, ws.b16,
                                 dev, s);
    }
    if (e != cudaSuccess)
        return cuda_fail(e, "preparation launch");
    GemmProblem p;
    p.a = ws.a16;
    p.b = b16;
    p.M = M;
    p.N = N;
    p.K = K;
    p.x_scale = ws.xs;
    p.w_scale = w_scale;
    p.bias = bias;
    p.scalar_scales = mode == CK_TENSORWISE;
    p.y = y;
    p.residual = residual;
    p.out_dtype = out_dtype;
    p.tail = graph ? nullptr : ws.tail;  // no K-split tail under capture
    std::string why;
    {
        ProfScope ps(kProfGemm, 1, s);
        e = launch_gemm(p, dev, s, &why);
    }
    if (e != cudaSuccess)
        return why.empty() ? cuda_fail(e, "GEMM launch") : fail(CK_ERR_CUDA, "%s", why.c_str());
    return CK_OK;
}

int ck_int8_linear(const void* x, const int8_t* w, const float* w_scale, const void* bias, const void* residual,
                   void* y, int64_t M, int64_t N, int64_t K, int mode, int out_dtype, void* workspace,
                   size_t workspace_bytes, void* stream)
{
    return linear_impl("int8_linear", true, x, w, nullptr, w_scale, bias, residual, y, M, N, K, mode, out_dtype, workspace,
                       workspace_bytes, stream);
}

int ck_int8_weight_codes(const int8_t* w, int64_t N, int64_t K, void* w_codes, void* stream)
{
    if (N < 0 || K <= 0 || K % 16 != 0)
        return fail(CK_ERR_INVALID_ARG, "N must be >= 0 and K a positive multiple of 16 (got N=%lld K=%lld)",
                    (long long)N, (long long)K);
    if (N > kMaxDim)
        return fail(CK_ERR_INVALID_ARG, "N must be < 2^31 (got %lld)", (long long)N);
    if (N == 0)
        return CK_OK;
    CK_REQUIRE_PTR(w);
    CK_REQUIRE_PTR(w_codes);
    DeviceInfo dev;
    int st = check_device(&dev);
    if (st != CK_OK)
        return st;
    cudaError_t e;
    {
        ProfScope ps(kProfWiden, 1, static_cast<cudaStream_t>(stream));
        e = launch_widen_int8(w, w_codes, N * K, dev, static_cast<cudaStream_t>(stream));
    }
    return e == cudaSuccess ? CK_OK : cuda_fail(e, "ck_int8_weight_codes launch");
}

size_t ck_int8_linear_codes_workspace_size(int64_t M, int64_t N, int64_t K, int mode)
{
    if (M < 0 || N < 0 || K < 0)
        return 0;
    return linear_ws_bytes(M, N, K, mode, kMaxPartials, false);
}

int ck_int8_linear_codes(const void* x, const void* w_codes, const float* w_scale, const void* bias,
                         const void* residual, void* y, int64_t M, int64_t N, int64_t K, int mode, int out_dtype,
                         void* workspace, size_t workspace_bytes, void* stream)
{
    return linear_impl("int8_linear_codes", false, x, nullptr, w_codes, w_scale, bias, residual, y, M, N, K, mode, out_dtype,
                       workspace, workspace_bytes, stream);
}

// ---- the 16-bit-activation path --------------------------------------------------
static size_t w8a16_ws_bytes(int64_t M, int64_t N, int64_t K, int mode)
{
    return align_up((size_t)N * K * 2) + (mode == CK_CONVROT ? align_up((size_t)M * K * 2) : 0);
}

size_t ck_w8a16_linear_workspace_size(int64_t M, int64_t N, int64_t K, int mode)
{
    if (M < 0 || N < 0 || K < 0)
        return 0;
    return w8a16_ws_bytes(M, N, K, mode);
}

int ck_w8a16_linear(const void* x, const int8_t* w, const float* w_scale, const void* bias, const void* residual,
                    void* y, int64_t M, int64_t N, int64_t K, int mode, int out_dtype, void* workspace,
                    size_t workspace_bytes, void* stream)
{
    if (mode != CK_TENSORWISE && mode != CK_PER_ROW && mode != CK_CONVROT)
        return fail(CK_ERR_INVALID_ARG, "mode must be 0 (tensorwise), 1 (per-row) or 2 (ConvRot), got %d", mode);
    if (!valid_out_dtype(out_dtype))
        return fail(CK_ERR_INVALID_ARG, "out_dtype must be 0 (bf16), 1 (fp16) or 2 (fp32), got %d", out_dtype);
    int st = check_gemm_shape(M, N, K);
    if (st != CK_OK)
        return st;
    if (mode == CK_CONVROT && K % 128 != 0)
        return fail(CK_ERR_INVALID_ARG, "ConvRot needs K % 128 == 0 (got %lld)", (long long)K);
    if (M == 0)
        return CK_OK;  // empty batch: x and y may be NULL
    CK_REQUIRE_PTR(x);
    CK_REQUIRE_PTR(w);
    CK_REQUIRE_PTR(w_scale);
    CK_REQUIRE_PTR(y);
    CK_REQUIRE_PTR(workspace);
    if (bias != nullptr && !aligned16(bias))
        return fail(CK_ERR_INVALID_ARG, "bias must be 16-byte aligned");
    if (residual != nullptr && !aligned16(residual))
        return fail(CK_ERR_INVALID_ARG, "residual must be 16-byte aligned");
    const size_t need = w8a16_ws_bytes(M, N, K, mode);
    if (workspace_bytes < need)
        return fail(CK_ERR_INVALID_ARG, "workspace too small: %zu bytes given, %zu needed", workspace_bytes, need);
    DeviceInfo dev;
    if ((st = check_device(&dev)) != CK_OK)
        return st;
    if (log_enabled())
        log_shape("w8a16_linear", M, N, K, mode,
                  std::string(mode == CK_CONVROT ? "rotate + widen" : "widen") +
                      " (1 launch) + tcgen05 bf16 GEMM with an fp32 sum over K, " +
                      describe_gemm_plan(M, N, K, true, false, dev));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t* p8 = static_cast<uint8_t*>(workspace);
    void* b16 = p8;
    void* a16 = p8 + align_up((size_t)N * K * 2);
    cudaError_t e;
    if (mode == CK_CONVROT) {
        ProfScope ps(kProfQuantize, 1, s);
        e = launch_rotate_bf16(x, M, K, a16, w, N * K, b16, dev, s);
    } else {
        ProfScope ps(kProfWiden, 1, s);
        e = launch_widen_int8(w, b16, N * K, dev, s);
    }
    if (e != cudaSuccess)
        return cuda_fail(e, "w8a16_linear operand launch");
    GemmProblem p;
    p.a = mode == CK_CONVROT ? a16 : x;
    p.b = b16;
    p.M = M;
    p.N = N;
    p.K = K;
    p.x_scale = nullptr;
    p.w_scale = w_scale;
    p.bias = bias;
    p.scalar_scales = mode == CK_TENSORWISE;
    p.y = y;
    p.residual = residual;
    p.out_dtype = out_dtype;
    p.mixed = true;
    std::string why;
    {
        ProfScope ps(kProfGemm, 1, s);
        e = launch_gemm(p, dev, s, &why);
    }
    if (e != cudaSuccess)
        return why.empty() ? cuda_fail(e, "w8a16_linear GEMM launch") : fail(CK_ERR_CUDA, "%s", why.c_str());
    return CK_OK;
}

int ck_convrot_prepare_weight(const float* W, int64_t N, int64_t K, int8_t* w, float* w_scale, void* stream)
{
    if (N < 0 || K <= 0)
        return fail(CK_ERR_INVALID_ARG, "N must be >= 0 and K >= 1 (got N=%lld K=%lld)", (long long)N, (long long)K);
    if (K % 128 != 0)
        return fail(CK_ERR_INVALID_ARG, "the ConvRot rotation needs K % 128 == 0 (got %lld)", (long long)K);
    if (N > kMaxDim)
        return fail(CK_ERR_INVALID_ARG, "N must be < 2^31 (got %lld)", (long long)N);
    if (N == 0)
        return CK_OK;
    CK_REQUIRE_PTR(W);
    CK_REQUIRE_PTR(w);
    CK_REQUIRE_PTR(w_scale);
    DeviceInfo dev;
    int st = check_device(&dev);
    if (st != CK_OK)
        return st;
    log_shape("convrot_prepare_weight", 0, N, K, CK_CONVROT, "rows-fwht");
    cudaError_t e = launch_convrot_weight(W, N, K, w, w_scale, dev, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? CK_OK : cuda_fail(e, "ck_convrot_prepare_weight launch");
}

size_t ck_int8_gemm_workspace_size(int64_t M, int64_t N, int64_t K)
{
    if (M < 0 || N < 0 || K < 0)
        return 0;
    return gemm_ws_bytes(M, N, K);
}

static int gemm_entry(const int8_t* q, const float* x_scale, const int8_t* w, const float* w_scale, const void* bias,
                      const void* residual, void* y, int32_t* acc, int64_t M, int64_t N, int64_t K,
                      int scalar_scales, int out_dtype, void* workspace, size_t workspace_bytes, void* stream,
                      const char* name)
{
    if (acc == nullptr && !valid_out_dtype(out_dtype))
        return fail(CK_ERR_INVALID_ARG, "out_dtype must be 0 (bf16), 1 (fp16) or 2 (fp32), got %d", out_dtype);
    int st = check_gemm_shape(M, N, K);
    if (st != CK_OK)
        return st;
    if (M == 0)
        return CK_OK;  // empty batch: q, x_scale, y / acc may be NULL
    CK_REQUIRE_PTR(q);
    CK_REQUIRE_PTR(w);
    CK_REQUIRE_PTR(workspace);
    if (acc == nullptr) {
        CK_REQUIRE_PTR(x_scale);
        CK_REQUIRE_PTR(w_scale);
        CK_REQUIRE_PTR(y);
        if (bias != nullptr && !aligned16(bias))
            return fail(CK_ERR_INVALID_ARG, "bias must be 16-byte aligned");
        if (residual != nullptr && !aligned16(residual))
            return fail(CK_ERR_INVALID_ARG, "residual must be 16-byte aligned");
    } else {
        CK_REQUIRE_PTR(acc);
    }
    const size_t need = gemm_ws_bytes(M, N, K);
    if (workspace_bytes < need)
        return fail(CK_ERR_INVALID_ARG, "workspace too small: %zu bytes given, %zu needed", workspace_bytes, need);
    DeviceInfo dev;
    if ((st = check_device(&dev)) != CK_OK)
        return st;
    if (M == 0)
        return CK_OK;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (log_enabled())
        log_shape(name, M, N, K, scalar_scales ? CK_TENSORWISE : CK_PER_ROW,
                  "widen (1 launch) + tcgen05 bf16-exact GEMM, " +
                      describe_gemm_plan(M, N, K, false, !stream_capturing(s), dev));
    uint8_t* p8 = static_cast<uint8_t*>(workspace);
    void* a16 = p8;
    void* b16 = p8 + align_up((size_t)M * K * 2);
    void* tail = static_cast<uint8_t*>(b16) + align_up((size_t)N * K * 2);
    cudaError_t e;
    {
        ProfScope ps(kProfWiden, 1, s);
        e = launch_widen2(q, M * K, a16, w, N * K, b16, dev, s);
    }
    if (e != cudaSuccess)
        return cuda_fail(e, "operand widening launch");
    GemmProblem p;
    p.a = a16;
    p.b = b16;
    p.M = M;
    p.N = N;
    p.K = K;
    p.x_scale = x_scale;
    p.w_scale = w_scale;
    p.bias = bias;
    p.scalar_scales = scalar_scales != 0;
    p.y = acc ? nullptr : y;
    p.residual = acc ? nullptr : residual;
    p.out_dtype = out_dtype;
    p.acc = acc;
    p.tail = stream_capturing(s) ? nullptr : tail;  // no K-split tail under capture
    std::string why;
    {
        ProfScope ps(kProfGemm, 1, s);
        e = launch_gemm(p, dev, s, &why);
    }
    if (e != cudaSuccess)
        return why.empty() ? cuda_fail(e, "GEMM launch") : fail(CK_ERR_CUDA, "%s", why.c_str());
    return CK_OK;
}

int ck_int8_gemm_dequant(const int8_t* q, const float* x_scale, const int8_t* w, const float* w_scale,
                         const void* bias, const void* residual, void* y, int64_t M, int64_t N, int64_t K,
                         int scalar_scales, int out_dtype, void* workspace, size_t workspace_bytes, void* stream)
{
    return gemm_entry(q, x_scale, w, w_scale, bias, residual, y, nullptr, M, N, K, scalar_scales, out_dtype,
                      workspace, workspace_bytes, stream, "int8_gemm_dequant");
}

int ck_int8_gemm_s32(const int8_t* q, const int8_t* w, int32_t* acc, int64_t M, int64_t N, int64_t K,
                     void* workspace, size_t workspace_bytes, void* stream)
{
    return gemm_entry(q, nullptr, w, nullptr, nullptr, nullptr, nullptr, acc, M, N, K, 0, CK_OUT_BF16, workspace,
                      workspace_bytes, stream, "int8_gemm_s32");
}

int ck_profile_begin(int with_events)
{
    g_prof_on = true;
    g_prof_events = with_events != 0;
    for (int k = 0; k < kProfKinds; ++k)
        g_prof_counts[k] = 0;
    for (const ProfRec& r : g_prof_recs) {
        g_prof_pool.push_back(r.a);
        g_prof_pool.push_back(r.b);
    }
    g_prof_recs.clear();
    return CK_OK;
}

int ck_profile_end(double* ms, int64_t* launches, int nkinds)
{
    g_prof_on = false;
    if (nkinds < 0 || (nkinds > 0 && (ms == nullptr || launches == nullptr)))
        return fail(CK_ERR_INVALID_ARG, "ck_profile_end needs ms[] and launches[] of nkinds entries");
    for (int k = 0; k < nkinds; ++k) {
        ms[k] = 0.0;
        launches[k] = k < kProfKinds ? g_prof_counts[k] : 0;
    }
    int status = CK_OK;
    for (const ProfRec& r : g_prof_recs) {
        float t = 0.0f;
        cudaError_t e = cudaEventSynchronize(r.b);
        if (e == cudaSuccess)
            e = cudaEventElapsedTime(&t, r.a, r.b);
        if (e != cudaSuccess && status == CK_OK)
            status = cuda_fail(e, "reading profile events");
        if (r.kind < nkinds)
            ms[r.kind] += t;
        g_prof_pool.push_back(r.a);
        g_prof_pool.push_back(r.b);
    }
    g_prof_recs.clear();
    return status;
}

int ck_gemm_tile_config(int64_t M, int64_t N, int64_t K, int* bn, int* cta_pair, int64_t* resident_units,
                        int* k_split)
{
    int st = check_gemm_shape(M, N, K);
    if (st != CK_OK)
        return st;
    CK_REQUIRE_PTR(bn);
    CK_REQUIRE_PTR(cta_pair);
    DeviceInfo dev;
    if ((st = check_device(&dev)) != CK_OK)
        return st;
    GemmPlan plan;
    cudaError_t e = plan_gemm(std::max<int64_t>(M, 1), N, K, false, dev, &plan);
    if (e != cudaSuccess)
        return cuda_fail(e, "GEMM planning");
    *bn = plan.bn;
    *cta_pair = plan.pair ? 1 : 0;
    if (resident_units)
        *resident_units = plan.resident;
    if (k_split)
        *k_split = plan.split;
    return CK_OK;
}

int ck_device_error(int clear)
{
    unsigned int v = 0;
    cudaError_t e = read_device_error(&v, clear != 0);
    if (e != cudaSuccess) {
        cuda_fail(e, "reading the device error word");
        return -1;
    }
    return (int)v;
}

int ck_selftest_wait_timeout(uint64_t timeout_ns, void* stream)
{
    DeviceInfo dev;
    int st = check_device(&dev);
    if (st != CK_OK)
        return st;
    unsigned int before = 0;
    cudaError_t e = read_device_error(&before, true);
    if (e != cudaSuccess)
        return cuda_fail(e, "clearing the device error word");
    if ((e = launch_wait_selftest(timeout_ns, static_cast<cudaStream_t>(stream))) != cudaSuccess)
        return cuda_fail(e, "wait self-test launch");
    unsigned int after = 0;
    if ((e = read_device_error(&after, true)) != cudaSuccess)
        return cuda_fail(e, "wait self-test");
    if (after & 16u)  // kErrWaitSelfTest
        return fail(CK_ERR_TIMEOUT, "the self-test wait gave up after %llu ns, as designed",
                    (unsigned long long)timeout_ns);
    return CK_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------------
// The layer with the activation and the output in host memory.
//
// The rows of the layer are independent (per-row and ConvRot scales are per row; the
// tensorwise scale needs all of x once, then the GEMM rows are again independent), so
// the call cuts M into slabs and overlaps, on three streams, the copy of slab i+1's
// activation into the device, the preparation and GEMM of slab i, and the copy of slab
// i-1's output back to the host.  Two device buffers alternate for the incoming
// activation and two for the outgoing output; events order each buffer's reuse.  The
// copies run on two internal streams per context (created on the first call there),
// the kernels on the caller's stream, which at the end waits for the last copy back: when
// the caller's stream has finished, y is complete in host memory.
namespace ck {
namespace {

struct HostLayout {
    int64_t R;          // rows per slab
    size_t x_slab, y_slab;
    size_t off_x[2], off_y[2], off_a16, off_xs, off_scratch, off_b16, off_tail, total;
};

int64_t host_slab_rows(int64_t M, int64_t N, int out_dtype, int64_t slab_rows)
{
    if (slab_rows > 0)
        return std::min<int64_t>(slab_rows, std::max<int64_t>(M, 1));
    // about 64 MB of output per slab, in whole 256-row tile pairs: against 256 MB the
    // pipeline fills and drains sooner (median steps on GB300: 80666x28672x5376 25.47 ->
    // 24.93 ms, 25900x16384x4096 5.34 -> 4.82 ms; the copy back to the host bounds both)
    const int64_t osize = out_dtype == CK_OUT_F32 ? 4 : 2;
    int64_t r = ((int64_t)64 << 20) / std::max<int64_t>(1, N * osize);
    r = std::max<int64_t>(256, r / 256 * 256);
    return std::min<int64_t>(r, std::max<int64_t>(M, 1));
}

HostLayout host_layout(int64_t M, int64_t N, int64_t K, int mode, int out_dtype, int64_t slab_rows)
{
    HostLayout L;
    L.R = host_slab_rows(M, N, out_dtype, slab_rows);
    const int64_t osize = out_dtype == CK_OUT_F32 ? 4 : 2;
    const bool tw = mode == CK_TENSORWISE;
    // tensorwise keeps all of x and its codes on the device (one scale for the tensor)
    L.x_slab = align_up((size_t)(tw ? M : L.R) * K * 2);
    L.y_slab = align_up((size_t)L.R * N * osize);
    size_t o = 0;
    L.off_x[0] = o;
    o += L.x_slab;
    L.off_x[1] = tw ? L.off_x[0] : o;
    if (!tw)
        o += L.x_slab;
    L.off_a16 = o;
    o += L.x_slab;
    L.off_xs = o;
    o += align_up(sizeof(float) * (size_t)(tw ? 1 : L.R));
    L.off_scratch = o;
    o += align_up(prep_tensorwise_scratch_bytes(kMaxPartialsForLayout));
    L.off_b16 = o;
    o += align_up((size_t)N * K * 2);
    L.off_y[0] = o;
    o += L.y_slab;
    L.off_y[1] = o;
    o += L.y_slab;
    L.off_tail = o;
    o += align_up(gemm_tail_bytes(L.R, N));
    L.total = o;
    return L;
}

// The two copy streams of the current context and the events that order the buffers.
struct HostPipe {
    cudaStream_t in = nullptr, out = nullptr;
    cudaEvent_t start, done, x_ready[2], x_free[2], y_ready[2], y_free[2];
    std::mutex* mu = nullptr;
};

cudaError_t host_pipe(HostPipe* out)
{
    static ContextCache<HostPipe> cache;
    return cache.get(out, [](HostPipe* p) {
        cudaError_t e = cudaStreamCreateWithFlags(&p->in, cudaStreamNonBlocking);
        if (e == cudaSuccess)
            e = cudaStreamCreateWithFlags(&p->out, cudaStreamNonBlocking);
        cudaEvent_t* evs[] = {&p->start, &p->done, &p->x_ready[0], &p->x_ready[1], &p->x_free[0],
                              &p->x_free[1],  &p->y_ready[0], &p->y_ready[1], &p->y_free[0], &p->y_free[1]};
        for (cudaEvent_t* ev : evs)
            if (e == cudaSuccess)
                e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
        p->mu = new std::mutex();
        return e;
    });
}

}  // namespace
}  // namespace ck

extern "C" size_t ck_int8_linear_host_workspace_size(int64_t M, int64_t N, int64_t K, int mode, int out_dtype,
                                                      int64_t slab_rows)
{
    if (M < 0 || N < 0 || K < 0 || slab_rows < 0)
        return 0;
    return host_layout(M, N, K, mode, out_dtype, slab_rows).total;
}

extern "C" int ck_int8_linear_host(const void* x_host, const int8_t* w, const float* w_scale, const void* bias,
                                   void* y_host, int64_t M, int64_t N, int64_t K, int mode, int out_dtype,
                                   int64_t slab_rows, void* workspace, size_t workspace_bytes, void* stream)
{
    if (mode != CK_TENSORWISE && mode != CK_PER_ROW && mode != CK_CONVROT)
        return fail(CK_ERR_INVALID_ARG, "mode must be 0 (tensorwise), 1 (per-row) or 2 (ConvRot), got %d", mode);
    if (!valid_out_dtype(out_dtype))
        return fail(CK_ERR_INVALID_ARG, "out_dtype must be 0 (bf16), 1 (fp16) or 2 (fp32), got %d", out_dtype);
    int st = check_gemm_shape(M, N, K);
    if (st != CK_OK)
        return st;
    if (mode == CK_CONVROT && K % 128 != 0)
        return fail(CK_ERR_INVALID_ARG, "ConvRot needs K % 128 == 0 (got %lld)", (long long)K);
    if (slab_rows < 0)
        return fail(CK_ERR_INVALID_ARG, "slab_rows must be >= 0 (0: chosen by the library)");
    if (M == 0)
        return CK_OK;
    CK_REQUIRE_PTR(x_host);
    CK_REQUIRE_PTR(w);
    CK_REQUIRE_PTR(w_scale);
    CK_REQUIRE_PTR(y_host);
    CK_REQUIRE_PTR(workspace);
    if (bias != nullptr && !aligned16(bias))
        return fail(CK_ERR_INVALID_ARG, "bias must be 16-byte aligned");
    const HostLayout L = host_layout(M, N, K, mode, out_dtype, slab_rows);
    if (workspace_bytes < L.total)
        return fail(CK_ERR_INVALID_ARG, "workspace too small: %zu bytes given, %zu needed", workspace_bytes, L.total);
    DeviceInfo dev;
    if ((st = check_device(&dev)) != CK_OK)
        return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (stream_capturing(s))
        return fail(CK_ERR_INVALID_ARG, "ck_int8_linear_host cannot be captured into a CUDA graph");
    HostPipe hp;
    cudaError_t e = host_pipe(&hp);
    if (e != cudaSuccess)
        return cuda_fail(e, "creating the copy streams");
    std::lock_guard<std::mutex> lock(*hp.mu);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    const uint8_t* xh = static_cast<const uint8_t*>(x_host);
    uint8_t* yh = static_cast<uint8_t*>(y_host);
    const bool tw = mode == CK_TENSORWISE;
    const int64_t osize = out_dtype == CK_OUT_F32 ? 4 : 2;
    const int64_t slabs = (M + L.R - 1) / L.R;
    float* xs = reinterpret_cast<float*>(ws + L.off_xs);
    void* a16 = ws + L.off_a16;
    void* b16 = ws + L.off_b16;
    if (log_enabled())
        log_shape("int8_linear_host", M, N, K, mode,
                  std::to_string(slabs) + " slabs of " + std::to_string(L.R) + " rows, copies on two streams");
#define CK_TRY(expr, what)                  \
    do {                                    \
        if ((e = (expr)) != cudaSuccess)    \
            return cuda_fail(e, what);      \
    } while (0)
    // the copy streams start after the work already on the caller's stream
    CK_TRY(cudaEventRecord(hp.start, s), "ck_int8_linear_host event");
    CK_TRY(cudaStreamWaitEvent(hp.in, hp.start, 0), "ck_int8_linear_host wait");
    CK_TRY(cudaStreamWaitEvent(hp.out, hp.start, 0), "ck_int8_linear_host wait");
    if (tw) {
        // all of x, then one preparation: the tensor's scale needs every value
        CK_TRY(cudaMemcpyAsync(ws + L.off_x[0], xh, (size_t)M * K * 2, cudaMemcpyHostToDevice, hp.in),
               "copying x to the device");
        CK_TRY(cudaEventRecord(hp.x_ready[0], hp.in), "ck_int8_linear_host event");
        CK_TRY(cudaStreamWaitEvent(s, hp.x_ready[0], 0), "ck_int8_linear_host wait");
        {
            ProfScope ps(kProfQuantize, 1, s);
            CK_TRY(launch_prep_tensorwise(ws + L.off_x[0], M, K, a16, xs, ws + L.off_scratch, kMaxPartialsForLayout, w,
                                          N * K, b16, dev, s),
                   "ck_int8_linear_host preparation launch");
        }
    }
    for (int64_t i = 0; i < slabs; ++i) {
        const int b = (int)(i & 1);
        const int64_t r0 = i * L.R;
        const int64_t rows = std::min<int64_t>(L.R, M - r0);
        if (!tw) {
            // activation slab in (after the preparation that last read this buffer)
            CK_TRY(cudaStreamWaitEvent(hp.in, hp.x_free[b], 0), "ck_int8_linear_host wait");
            CK_TRY(cudaMemcpyAsync(ws + L.off_x[b], xh + r0 * K * 2, (size_t)rows * K * 2, cudaMemcpyHostToDevice,
                                   hp.in),
                   "copying an x slab to the device");
            CK_TRY(cudaEventRecord(hp.x_ready[b], hp.in), "ck_int8_linear_host event");
            CK_TRY(cudaStreamWaitEvent(s, hp.x_ready[b], 0), "ck_int8_linear_host wait");
            ProfScope ps(kProfQuantize, 1, s);
            // the weight is widened once, by the first slab's launch
            CK_TRY(launch_prep_rows(ws + L.off_x[b], rows, K, mode == CK_CONVROT, a16, xs, i == 0 ? w : nullptr,
                                    N * K, b16, dev, s),
                   "ck_int8_linear_host preparation launch");
            CK_TRY(cudaEventRecord(hp.x_free[b], s), "ck_int8_linear_host event");
        }
        // the GEMM of the slab into an output buffer the previous copy back has released
        CK_TRY(cudaStreamWaitEvent(s, hp.y_free[b], 0), "ck_int8_linear_host wait");
        GemmProblem p;
        p.a = static_cast<uint8_t*>(a16) + (tw ? r0 * K * 2 : 0);
        p.b = b16;
        p.M = rows;
        p.N = N;
        p.K = K;
        p.x_scale = xs;
        p.w_scale = w_scale;
        p.bias = bias;
        p.scalar_scales = tw;
        p.y = ws + L.off_y[b];
        p.out_dtype = out_dtype;
        p.tail = ws + L.off_tail;
        std::string why;
        {
            ProfScope ps(kProfGemm, 1, s);
            e = launch_gemm(p, dev, s, &why);
        }
        if (e != cudaSuccess)
            return why.empty() ? cuda_fail(e, "ck_int8_linear_host GEMM launch") : fail(CK_ERR_CUDA, "%s", why.c_str());
        CK_TRY(cudaEventRecord(hp.y_ready[b], s), "ck_int8_linear_host event");
        // ... and the slab's output back to the host
        CK_TRY(cudaStreamWaitEvent(hp.out, hp.y_ready[b], 0), "ck_int8_linear_host wait");
        CK_TRY(cudaMemcpyAsync(yh + r0 * N * osize, ws + L.off_y[b], (size_t)rows * N * osize, cudaMemcpyDeviceToHost,
                               hp.out),
               "copying a y slab to the host");
        CK_TRY(cudaEventRecord(hp.y_free[b], hp.out), "ck_int8_linear_host event");
    }
    // the caller's stream completes only after the last copy back
    CK_TRY(cudaEventRecord(hp.done, hp.out), "ck_int8_linear_host event");
    CK_TRY(cudaStreamWaitEvent(s, hp.done, 0), "ck_int8_linear_host wait");
#undef CK_TRY
    return CK_OK;
}

// ---------------------------------------------------------------------------------
// Tensorwise quantize without any allocation.
//
// Some callers cannot allocate device memory at all.  A real-time inference loop may
// reserve its whole memory budget before it starts and forbid allocator traffic while it
// runs: an allocation can block, or fail on a fragmented heap, at a moment the loop
// cannot afford.  A host that embeds this library under its own memory manager must
// account for every byte on the device and hands out nothing per call, and a plugin
// loaded into such a host sees only the buffers it is given.  These callers can pass
// their inputs and outputs, but not a workspace.  For them the partial maxima of the
// tensorwise quantize live in a fixed array that is part of the loaded module itself.
//
// Costs and limits:
//   - the array holds kNoallocMaxPartials floats (16 KiB) on every GPU where this
//     library's module is loaded, for the life of the process;
//   - one partial maximum covers kNoallocValuesPerPartial input values, so M*K may be
//     at most kNoallocMaxPartials * kNoallocValuesPerPartial = 134,217,728 values;
//     larger tensors are rejected with CK_ERR_INVALID_ARG before anything is enqueued;
//   - every call uses the same array and it keeps the last call's contents.  Nothing in
//     it needs to start at zero: every slot a call reads was written earlier by that same
//     call.  But two calls whose kernels overlap on the GPU -- different streams, or
//     different host threads -- race on it and may return a wrong scale.  Serialize such
//     calls on one stream;
//   - the first call in a CUDA context looks up the array's device address there
//     (cudaGetSymbolAddress, with that context's device current; this also loads the
//     module on the device) and keeps it for later calls in the same context.  Make that
//     first call before any stream capture begins.  A device reset creates a new context,
//     whose first call looks the address up again.
namespace ck {
namespace {

constexpr int kNoallocMaxPartials = 4096;
constexpr int64_t kNoallocVectorsPerPartial = 4096;  // 16-byte vectors of 8 bf16
constexpr int64_t kNoallocValuesPerPartial = kNoallocVectorsPerPartial * 8;

static __device__ __align__(256) float g_noalloc_partials[kNoallocMaxPartials];

// Device address of g_noalloc_partials in the current context.  In host code the
// array's name is only a host-side stand-in, never a device address: a kernel given it
// would fault, or silently use the wrong memory where the GPU can reach host memory.
int noalloc_scratch(float** out)
{
    static ContextCache<float*> cache;
    const cudaError_t e = cache.get(out, [](float** p) {
        void* a = nullptr;
        const cudaError_t r = cudaGetSymbolAddress(&a, g_noalloc_partials);
        *p = static_cast<float*>(a);
        return r;
    });
    return e == cudaSuccess ? CK_OK : cuda_fail(e, "looking up the no-allocation scratch array");
}

}  // namespace
}  // namespace ck

extern "C" int ck_quantize_int8_tensorwise_noalloc(const void* x, int64_t M, int64_t K, int8_t* q, float* x_scale,
                                                   void* stream)
{
    if (M < 0 || K <= 0)
        return fail(CK_ERR_INVALID_ARG, "M must be >= 0 and K >= 1 (got M=%lld K=%lld)", (long long)M, (long long)K);
    if (K % 16 != 0)
        return fail(CK_ERR_INVALID_ARG, "K must be a multiple of 16 (got %lld)", (long long)K);
    if (M > 0 && M > (kNoallocMaxPartials * kNoallocValuesPerPartial) / K)
        return fail(CK_ERR_INVALID_ARG,
                    "M*K = %lld exceeds the no-allocation limit of %lld values (%d partial maxima of %lld values); "
                    "use ck_quantize_int8_tensorwise with a workspace",
                    (long long)M * (long long)K, (long long)(kNoallocMaxPartials * kNoallocValuesPerPartial),
                    kNoallocMaxPartials, (long long)kNoallocValuesPerPartial);
    if (M == 0)
        return CK_OK;
    CK_REQUIRE_PTR(x);
    CK_REQUIRE_PTR(q);
    CK_REQUIRE_PTR(x_scale);
    DeviceInfo dev;
    int st = check_device(&dev);
    if (st != CK_OK)
        return st;
    float* partials = nullptr;
    if ((st = noalloc_scratch(&partials)) != CK_OK)
        return st;
    const int64_t nvec = (M * K) >> 3;
    const int nparts = (int)((nvec + kNoallocVectorsPerPartial - 1) / kNoallocVectorsPerPartial);
    cudaError_t e = launch_quantize_tensorwise_parts(x, M, K, q, nullptr, x_scale, partials, nparts, dev,
                                                     static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? CK_OK : cuda_fail(e, "ck_quantize_int8_tensorwise_noalloc launch");
}
