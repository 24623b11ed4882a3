// gemm.cu -- exact INT8 x INT8 GEMM with the dequant epilogue fused, on the sm_103a
// tensor cores (tcgen05), persistent and warp-specialised.
//
// What it computes (comfy-kitchen issue #280, "Kernel used" and "Exactness"):
//   acc[m,n] = sum_k q[m,k] * w[n,k]   exactly (int32), then in fp32
//   y[m,n]   = bf16( ((float(acc) * x_scale[m]) * w_scale[n]) + bias[n] )
// with every address formed in 64 bits (issue #136, "Suggested fix").
//
// Engine.  sm_103a has no int8 tensor-core kind, so the int8 codes are fed to the
// bf16 kind (kind::f16) as bf16 values: every integer in [-127, 127] is a bf16 exactly,
// every product is an integer of magnitude <= 16129, and any partial sum of at most
// 1024 such products has magnitude <= 16,516,096 < 2^24, so it is an exact fp32 integer.
// The MMA therefore accumulates K in chunks of 1024 into an fp32 TMEM accumulator,
// restarting the accumulator at each chunk; the epilogue warps convert each finished
// chunk to int32 (exact) and add it to int32 running sums held in registers.  The
// int32 sum is the true accumulator; it never leaves the SM.
//
// CTA pairs (the default when there are at least two 128-row tiles).  A 2-CTA cluster
// computes a 256 x bn tile (bn a multiple of 32 up to 256, chosen per launch) with
// tcgen05 cta_group::2: each CTA holds 128 activation rows and bn/2 of the weight rows of
// every k-block in its own shared memory, the leader CTA issues 256 x bn x 16 MMAs that
// read both CTAs' operands, and each CTA's TMEM receives its own 128 output rows.  Per SM
// this halves the weight bytes that shared memory must take in and hand to the tensor
// core, compared with one CTA per 128 x bn tile.  Problems with a single tile row (and
// one-wave problems the planner prices cheaper so) run one CTA per 128 x bn tile.
//
// Roles (one CTA per SM, 12 warps):
//   warp 0      TMA producer: per k-block this CTA's A rows and B rows as 64-deep bf16
//               boxes into a ring of 128B-swizzled stages -- CTA pairs stage 128-deep
//               k-blocks (two boxes per operand, three stages), single CTAs 64-deep ones
//               (four stages); in a pair, completion is counted on the leader's barrier;
//   warp 1      allocates 512 TMEM columns (two fp32 accumulators of 256 columns) and, in
//               the leader (or single CTA), issues the MMAs from one thread;
//   warps 2-3   idle (they complete warpgroup 0 for the register re-balancing);
//   warps 4-11  epilogue: warp w reads TMEM lanes 32*(w%4).. and one 128-column half;
//               drains each chunk into its running sums, then dequantizes, converts to
//               the output type, stages 32-row boxes in shared memory and stores them
//               with TMA.
// The two accumulators ping-pong, so the MMA of the next chunk (or tile) overlaps the
// drain and the store of the previous one.  Tiles are visited in a grouped order
// (group_m unit rows share a sweep over N) so concurrently resident CTAs reuse operands
// from L2.  Every wait is bounded (see mbar_wait); a timed-out CTA records an error bit,
// lets its copies and MMAs finish, frees TMEM and exits.
#include <algorithm>
#include <atomic>
#include <chrono>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include <unistd.h>

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "ck_device.cuh"
#include "ck_internal.h"
#include "gemm_common.cuh"

namespace ck {

__device__ unsigned int g_device_error;

namespace gemm {

constexpr int BM = 128;       // rows of a CTA's tile (a pair covers 2 * BM)
constexpr int BN = 256;       // widest tile; a launch may use any multiple of 32 up to it
constexpr int BK = 64;        // one 128-byte swizzle row of bf16: the width of every TMA box
constexpr int UMMA_K = 16;    // K per kind::f16 instruction
static_assert(BK / UMMA_K == 4, "mma_bf16_kblock issues the four MMAs of a 64-deep sub-block");
constexpr int CHUNK_K = 1024; // products per exact fp32 chunk
constexpr int EPI_WARPS = 8;
constexpr int EPI_WARP0 = 4;                  // warps 0-3: producer, MMA issuer, two idle
constexpr int THREADS = 32 * (EPI_WARP0 + EPI_WARPS);
// Registers per thread after the warpgroups re-balance (setmaxnreg): the first
// warpgroup needs few, the two epilogue warpgroups hold 128 running sums per thread.
// The launch must provide at least their sum (checked on the host before launching).
constexpr uint32_t REGS_WG0 = 56;
constexpr uint32_t REGS_EPI = 216;
constexpr uint32_t REGS_NEEDED_PER_BLOCK = 128 * REGS_WG0 + 256 * REGS_EPI;
constexpr uint32_t A_BYTES = BM * BK * 2;
constexpr int B_BOX_ROWS = BN / 2;                       // most weight rows per TMA box
constexpr uint32_t B_BOX_BYTES = B_BOX_ROWS * BK * 2;
constexpr uint32_t OUT_BYTES = EPI_WARPS * 2 * OUT_BUF_BYTES;
constexpr uint32_t TMEM_COLS = 2 * BN;
constexpr uint32_t BAR_BYTES = 256;

// Per-mode shapes: a pair CTA stages 128 weight rows per 64-deep sub-block, a single CTA
// 256.  A pipeline stage (k-block) holds KSUB sub-blocks: every stage costs a fixed
// hand-off (barriers, loads, commit) that 64-deep stages could not hide -- a unit's
// k-block took ~305 ns however narrow the tile; CTA pairs stage 128-deep k-blocks (three
// stages), 4096^3 went from 96 to 80 us.  Single CTAs stage twice the weight rows, so a
// 128-deep stage leaves them two stages, which was slower: they keep 64-deep ones.
template <bool PAIR>
struct Mode {
    static constexpr int KSUB = PAIR ? 2 : 1;
    static constexpr int KB = BK * KSUB;                  // K per k-block
    static constexpr int CHUNK_KB = CHUNK_K / KB;         // k-blocks per exact fp32 chunk
    static constexpr uint32_t B_BYTES = PAIR ? B_BOX_BYTES : 2 * B_BOX_BYTES;  // per sub-block
    // a stage: the KSUB A sub-blocks, then the KSUB B sub-blocks
    static constexpr uint32_t STAGE_BYTES = KSUB * (A_BYTES + B_BYTES);
    static constexpr int STAGES = PAIR ? 3 : 4;
    static constexpr uint32_t IDESC_M = PAIR ? idesc_bf16_f32<2 * BM, 0>() : idesc_bf16_f32<BM, 0>();
    static constexpr size_t SMEM_BYTES = 1024 + (size_t)STAGES * STAGE_BYTES + OUT_BYTES + BAR_BYTES;
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
    static_assert((2 * STAGES + 5) * 8 + 8 <= BAR_BYTES, "barrier area");
};

struct Args {
    int64_t M, N, K;
    const float* xs;
    const float* ws;
    const __nv_bfloat16* bias;
    const void* residual;   // [M,N] of the output type, added after the bias; may alias y
    int32_t* acc;
    int64_t num_units;      // pair-tiles (pairs) or tiles
    int unit_rows;          // tile rows per unit: 2 (pairs) or 1
    int bn;                 // tile width in N (multiple of 32, <= BN)
    uint32_t idesc;         // MMA instruction descriptor for this width
    uint32_t tx_bytes;      // bytes of one k-block counted on the (leader's) full barrier
    int units_m, tiles_m, tiles_n, num_kb, group_m;
    int scalar_scales;
    float one;              // 1.0f, a value the compiler cannot see (the epilogue's packed adds)
    int chunk_kb;           // k-blocks per TMEM accumulation: 1024 products (exact), all of K (16-bit activations)
    uint64_t timeout_ns;
    // K-split of the last partial wave: units [full_units, num_units) are each computed
    // as `split` K-slices by different units of the grid; every slice writes its int32
    // running sums to `partials`, and the slice that arrives last at the unit's counter
    // in `tail_slots` adds the others' sums and runs the epilogue.
    int64_t full_units;
    int64_t num_items;      // full_units + (num_units - full_units) * split
    int split;              // 1 = no split
    int32_t* partials;      // [tail unit][slice][rank][epilogue warp][column group of 4][lane][4] int32
    unsigned long long* tail_slots;  // [tail unit][rank][epilogue warp] (tag << 16) | arrivals, 16 bytes apart
    unsigned long long epoch;        // this launch's tag for tail_slots
};

// One work item of the persistent loop: a whole unit, or one K-slice of a tail unit.
struct Item {
    int64_t unit;
    int64_t tail;   // index among the tail units (slice >= 0 only)
    int kb_begin, kb_end;
    int slice;      // -1: the whole K range
};

template <bool SPLIT>
__device__ __forceinline__ Item item_of(int64_t it, const Args& a)
{
    Item r;
    if (!SPLIT || it < a.full_units) {
        r.unit = it;
        r.tail = 0;
        r.kb_begin = 0;
        r.kb_end = a.num_kb;
        r.slice = -1;
    } else {
        const int64_t j = it - a.full_units;
        r.tail = j / a.split;
        r.slice = (int)(j - r.tail * a.split);
        r.unit = a.full_units + r.tail;
        r.kb_begin = (int)((int64_t)a.num_kb * r.slice / a.split);
        r.kb_end = (int)((int64_t)a.num_kb * (r.slice + 1) / a.split);
    }
    return r;
}

// Count one arrival at a tail unit's 64-bit slot, packed as (launch tag << 16) | count:
// a slot still tagged by an earlier launch (or holding anything else) restarts at 1.
// The tag is the launch's 64-bit epoch cut to 48 bits, so stale or random slot contents
// match it with probability 2^-48.  Returns true for the arrival that makes the count
// `split`.  Each failed swap means another arrival went in (or the first read was
// stale), so the retries are bounded.
__device__ __forceinline__ bool tail_arrive(unsigned long long* slot, unsigned long long epoch, int split,
                                            unsigned int* err)
{
    const unsigned long long tag = epoch & 0xFFFFFFFFFFFFull;
    unsigned long long old = __ldcg(slot);
    for (int i = 0; i < 4 * split + 8; ++i) {
        const unsigned long long count = (old >> 16) == tag ? (old & 0xFFFFull) + 1 : 1;
        const unsigned long long prev = atomicCAS(slot, old, (tag << 16) | count);
        if (prev == old)
            return count == (unsigned long long)split;
        old = prev;
    }
    atomicOr(err, kErrTailCount);
    return false;
}

// Unit u (a pair-tile, or a tile) -> (unit row, tile column) in grouped order.
__device__ __forceinline__ void unit_coords(int64_t u, const Args& a, int& um, int& nb)
{
    const int64_t per_group = (int64_t)a.group_m * a.tiles_n;
    const int64_t g = u / per_group;
    const int64_t first = g * a.group_m;
    const int64_t rows = min((int64_t)a.group_m, (int64_t)a.units_m - first);
    const int64_t r = u - g * per_group;
    um = (int)(first + r % rows);
    nb = (int)(r / rows);
}

// 12 warps put three warps on each of the four SM sub-partitions, whose register files
// hold 16K registers each: at most 168 registers per thread at launch, re-balanced to
// REGS_WG0 / REGS_EPI once the roles split (32 x (56 + 2 x 216) <= 16K per
// sub-partition as well).
// MIXED: 16-bit activations times int8 weight codes (both bf16 operands), the fp32
// accumulation over all of K kept in TMEM, epilogue (sum * w_scale) + bias.
// SPLIT: the launch splits its last partial wave along K; RES: a residual is added.
// Both live only in their own instances: unused code in the common kernel measurably
// slowed it (instruction fetch on the first tile, register allocation).
template <bool RAW, bool PAIR, int OUT, bool MIXED, bool SPLIT, bool RES>
__global__ void __launch_bounds__(THREADS, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmY, const Args args)
{
    using MD = Mode<PAIR>;
    constexpr int STAGES = MD::STAGES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* s_ab = smem;
    uint8_t* s_out = smem + (size_t)STAGES * MD::STAGE_BYTES;
    uint64_t* bars = reinterpret_cast<uint64_t*>(s_out + OUT_BYTES);
    uint64_t* full = bars;
    uint64_t* empty = bars + STAGES;
    uint64_t* acc_full = bars + 2 * STAGES;
    uint64_t* acc_empty = acc_full + 2;
    uint64_t* drain = acc_empty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    unsigned int* err = &g_device_error;
    const int rank = PAIR ? (int)cluster_ctarank() : 0;  // 0 = leader: issues the MMAs
    const bool leader = rank == 0;
    const int cluster = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
    const int clusters = PAIR ? (int)(gridDim.x >> 1) : (int)gridDim.x;
    constexpr uint16_t kPairMask = 0x3;

    if (warp == 0 && lane == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], PAIR ? 2 * EPI_WARPS : EPI_WARPS);  // pair: both CTAs' epilogues
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
        fence_proxy_async_smem();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        if (!RAW)
            tma_prefetch_desc(&tmY);
    }
    if (warp == 1) {
        if (PAIR) {
            tmem_alloc_pair(tmem_slot, TMEM_COLS);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(tmem_slot, TMEM_COLS);
            tmem_relinquish();
        }
    }
    __syncwarp();  // reconverge warps 0 and 1 after their one-lane / one-warp set-up
    tc_fence_before();
    if (PAIR)
        cluster_sync();  // both CTAs' barriers and TMEM exist before either is used
    else
        __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // everything above overlapped the previous kernel; from here on global memory is read
    griddep_wait();
    if (warp < EPI_WARP0) {
        // ---------------------------------------------------------------- warpgroup 0
        setmaxnreg_dec<REGS_WG0>();
        if (warp == 0) {
            // ------------------------------------------------------------ TMA producer
            if (lane == 0) {
                int stage = 0;
                uint32_t phase = 0;
                uint32_t issued_mask = 0;       // stages holding a load
                uint32_t issued_parity = 0;     // parity of that load's phase, per stage
                bool ok = true;
                for (int64_t it = cluster; ok && it < args.num_items; it += clusters) {
                    const Item w = item_of<SPLIT>(it, args);
                    int um, nb;
                    unit_coords(w.unit, args, um, nb);
                    const int32_t m0 = (um * args.unit_rows + rank) * BM, n0 = nb * args.bn;
                    const int half_rows = args.bn >> 1;  // weight rows per box
                    for (int kb = w.kb_begin; kb < w.kb_end; ++kb) {
                        if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, err, kErrWaitProducer, args.timeout_ns)) {
                            ok = false;
                            break;
                        }
                        uint8_t* sa = s_ab + (size_t)stage * MD::STAGE_BYTES;
                        uint8_t* sb = sa + MD::KSUB * A_BYTES;
                        if (PAIR) {
                            // both CTAs' bytes are counted on the leader's barrier
                            const uint32_t bar = mapa_shared(&full[stage], 0);
                            if (leader)
                                mbar_arrive_expect_tx(&full[stage], args.tx_bytes);
#pragma unroll
                            for (int sub = 0; sub < MD::KSUB; ++sub) {
                                const int32_t k0 = kb * MD::KB + sub * BK;
                                tma_load_2d_pair(sa + sub * A_BYTES, &tmA, bar, k0, m0);
                                tma_load_2d_pair(sb + sub * MD::B_BYTES, &tmB, bar, k0, n0 + rank * half_rows);
                            }
                        } else {
                            mbar_arrive_expect_tx(&full[stage], args.tx_bytes);
#pragma unroll
                            for (int sub = 0; sub < MD::KSUB; ++sub) {
                                const int32_t k0 = kb * MD::KB + sub * BK;
                                uint8_t* b = sb + sub * MD::B_BYTES;
                                tma_load_2d(sa + sub * A_BYTES, &tmA, &full[stage], k0, m0);
                                tma_load_2d(b, &tmB, &full[stage], k0, n0);
                                tma_load_2d(b + half_rows * BK * 2, &tmB, &full[stage], k0, n0 + half_rows);
                            }
                        }
                        issued_mask |= 1u << stage;
                        issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                        if (++stage == STAGES) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                }
                if (!ok && leader) {
                    // the CTA is aborting: let every issued copy land before shared memory is
                    // released (the leader's barriers count both CTAs' bytes)
                    for (int s = 0; s < STAGES; ++s)
                        if (issued_mask & (1u << s))
                            drain_wait(&full[s], (issued_parity >> s) & 1u, err, args.timeout_ns);
                }
            }
            __syncwarp();  // reconverge before the block-wide barrier below
        } else if (warp == 1) {
            // ------------------------------------------------------------ MMA issuer
            if (lane == 0 && leader) {
                int stage = 0;
                uint32_t phase = 0;
                uint32_t acc_iter = 0;
                bool ok = true;
                // One thread issues every MMA, so its loop is kept short: the invariants live
                // in registers and a stage's descriptors are stage 0's plus an offset in the
                // address field (shared addresses >> 4 stay below 2^14: no carry leaves it).
                const uint32_t idesc = args.idesc;
                const int chunk_kb = args.chunk_kb;
                const uint64_t timeout_ns = args.timeout_ns;
                const uint64_t desc_a0 = desc_kmajor_sw128(smem_u32(s_ab));
                constexpr uint64_t kDescStage = MD::STAGE_BYTES >> 4;
                constexpr uint64_t kDescB = (MD::KSUB * A_BYTES) >> 4;
                for (int64_t it = cluster; ok && it < args.num_items; it += clusters) {
                    const Item w = item_of<SPLIT>(it, args);
                    for (int kb0 = w.kb_begin; kb0 < w.kb_end; kb0 += chunk_kb) {
                        const uint32_t buf = acc_iter & 1u;
                        const uint32_t acc_phase = (acc_iter >> 1) & 1u;
                        if (!mbar_wait(&acc_empty[buf], acc_phase ^ 1u, abort_flag, err, kErrWaitMma, timeout_ns)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t d_tmem = tmem_base + buf * BN;
                        const int kend = min(kb0 + chunk_kb, w.kb_end);
                        for (int kb = kb0; kb < kend; ++kb) {
                            if (!mbar_wait(&full[stage], phase, abort_flag, err, kErrWaitMma, timeout_ns)) {
                                ok = false;
                                break;
                            }
                            tc_fence_after();
                            const uint64_t ad = desc_a0 + (uint64_t)stage * kDescStage;
#pragma unroll
                            for (int sub = 0; sub < MD::KSUB; ++sub)
                                mma_bf16_kblock<PAIR>(d_tmem, ad + sub * (A_BYTES >> 4),
                                                      ad + kDescB + sub * (MD::B_BYTES >> 4), idesc,
                                                      (kb > kb0 || sub > 0) ? 1u : 0u);
                            if (PAIR)
                                mma_commit_pair(&empty[stage], kPairMask);  // frees the stage in both CTAs
                            else
                                mma_commit(&empty[stage]);
                            if (++stage == STAGES) {
                                stage = 0;
                                phase ^= 1u;
                            }
                        }
                        if (!ok)
                            break;
                        if (PAIR)
                            mma_commit_pair(&acc_full[buf], kPairMask);
                        else
                            mma_commit(&acc_full[buf]);
                        ++acc_iter;
                    }
                }
                // every MMA issued above must be complete before TMEM is released
                if (PAIR)
                    mma_commit_pair(drain, 0x1);
                else
                    mma_commit(drain);
                drain_wait(drain, 0, err, args.timeout_ns);
            }
            __syncwarp();  // reconverge before the block-wide barrier below
        }
    } else {
        // ---------------------------------------------------------------- epilogue
        setmaxnreg_inc<REGS_EPI>();
        const int e = warp - EPI_WARP0;
        const int quarter = warp & 3;  // TMEM lanes this warp may access
        const int half = e >> 2;       // which 128 of the 256 tile columns
        const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
        uint8_t* obuf = s_out + (size_t)e * 2 * OUT_BUF_BYTES;
        uint32_t acc_iter = 0;
        uint32_t nstore = 0;
        bool ok = true;
        for (int64_t it = cluster; ok && it < args.num_items; it += clusters) {
            const Item w = item_of<SPLIT>(it, args);
            int um, nb;
            unit_coords(w.unit, args, um, nb);
            const int64_t m0 = (int64_t)(um * args.unit_rows + rank) * BM;
            const int64_t n0 = (int64_t)nb * args.bn;
            // columns of the tile in this warp's half: a multiple of 32 in [0, 128]
            const int ncols = max(0, min(128, args.bn - half * 128));
            const int64_t row = m0 + quarter * 32 + lane;
            const int64_t cbase = n0 + half * 128;
            float xsv = 0.0f, ws_scalar = 0.0f;
            // w_scale and bias of columns cbase + 4 lane .. + 3 (0 past the tile or N); the store
            // loop takes a column's values from its lane by shuffle.  Loaded here, they are in
            // flight during the K loop: loaded per chunk in the store loop, their latency held
            // up every tile's stores, ~4 us per launch at 4096^3 (the last tile's is exposed).
            float wsr[4] = {0.0f, 0.0f, 0.0f, 0.0f}, bsr[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            if (!RAW) {  // the scalar scales and this lane's row scale, in flight during the K loop
                if (args.scalar_scales)
                    ws_scalar = __ldg(args.ws);
                if (!MIXED)
                    xsv = args.scalar_scales ? __ldg(args.xs) : (row < args.M ? __ldg(args.xs + row) : 0.0f);
                const int64_t c4 = cbase + 4 * lane;
                if (4 * lane < ncols && c4 < args.N) {  // N % 8 == 0: a group of 4 is all in or all out
                    if (!args.scalar_scales) {
                        const float4 w4 = __ldg(reinterpret_cast<const float4*>(args.ws + c4));
                        wsr[0] = w4.x;
                        wsr[1] = w4.y;
                        wsr[2] = w4.z;
                        wsr[3] = w4.w;
                    }
                    if (args.bias) {
                        const uint2 braw = __ldg(reinterpret_cast<const uint2*>(args.bias + c4));
                        const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&braw);
                        bsr[0] = __low2float(b2[0]);
                        bsr[1] = __high2float(b2[0]);
                        bsr[2] = __low2float(b2[1]);
                        bsr[3] = __high2float(b2[1]);
                    }
                }
            }
            int32_t run[128];
#pragma unroll
            for (int j = 0; j < 128; ++j)
                run[j] = 0;
            for (int kb0 = w.kb_begin; kb0 < w.kb_end; kb0 += args.chunk_kb) {
                const uint32_t buf = acc_iter & 1u;
                const uint32_t acc_phase = (acc_iter >> 1) & 1u;
                // one lane polls, the warp follows its verdict (keeps the warp converged
                // for the .sync.aligned TMEM loads)
                int got = 1;
                if (lane == 0)
                    got = mbar_wait(&acc_full[buf], acc_phase, abort_flag, err, kErrWaitEpilogue, args.timeout_ns);
                got = __shfl_sync(0xffffffffu, got, 0);
                if (!got) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t taddr = tmem_base + lane_base + buf * BN + half * 128;
#pragma unroll
                for (int g = 0; g < 8; ++g) {
                    if (g * 16 < ncols) {  // warp-uniform
                        uint32_t v[16];
                        tmem_ld_32x32b_x16(taddr + g * 16, v);
                        tmem_wait_ld();
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            if (MIXED)  // one chunk holds the whole fp32 sum: keep its bits
                                run[g * 16 + j] = (int32_t)v[j];
                            else
                                run[g * 16 + j] += __float2int_rz(__uint_as_float(v[j]));  // exact integer
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if (PAIR)
                        mbar_arrive_cluster(mapa_shared(&acc_empty[buf], 0));  // the leader's MMA waits on it
                    else
                        mbar_arrive(&acc_empty[buf]);
                }
                ++acc_iter;
            }
            if (!ok)
                break;

            if (SPLIT && w.slice >= 0 && ncols > 0) {
                // one K-slice of a tail unit: publish this warp's sums; the last slice to
                // arrive adds the others' and goes on to the epilogue
                constexpr int RANKS = PAIR ? 2 : 1;
                const int lslot = rank * EPI_WARPS + e;                       // this warp within the unit
                const int64_t wslot = w.tail * (RANKS * EPI_WARPS) + lslot;   // its arrival counter
                const int64_t span = (int64_t)RANKS * EPI_WARPS * 32 * 128;   // int32 per slice
                // a warp's sums are 32 column groups of 4, each stored as 32 lanes x 16 bytes
                // in a row, so every store and load of a warp covers 512 contiguous bytes
                int32_t* mine = args.partials + (w.tail * args.split + w.slice) * span + lslot * (32 * 128) + lane * 4;
#pragma unroll
                for (int c4 = 0; c4 < 32; ++c4)
                    if (4 * c4 < ncols)
                        __stcg(reinterpret_cast<int4*>(mine + c4 * 128),
                               make_int4(run[4 * c4], run[4 * c4 + 1], run[4 * c4 + 2], run[4 * c4 + 3]));
                __threadfence();
                __syncwarp();
                int last = 0;
                if (lane == 0)
                    last = tail_arrive(args.tail_slots + 2 * wslot, args.epoch, args.split, err) ? 1 : 0;
                last = __shfl_sync(0xffffffffu, last, 0);
                if (!last)
                    continue;  // another slice stores the unit
                __threadfence();  // the other slices' sums, published before their arrivals
                for (int sl = 0; sl < args.split; ++sl) {
                    if (sl == w.slice)
                        continue;
                    const int32_t* other =
                        args.partials + (w.tail * args.split + sl) * span + lslot * (32 * 128) + lane * 4;
#pragma unroll
                    for (int c4 = 0; c4 < 32; ++c4)
                        if (4 * c4 < ncols) {
                            const int4 v = __ldcg(reinterpret_cast<const int4*>(other + c4 * 128));
                            run[4 * c4] += v.x;
                            run[4 * c4 + 1] += v.y;
                            run[4 * c4 + 2] += v.z;
                            run[4 * c4 + 3] += v.w;
                        }
                }
            }

            if (RAW) {
                if (row < args.M) {
                    int32_t* dst = args.acc + row * args.N;
#pragma unroll
                    for (int c4 = 0; c4 < 32; ++c4) {
                        const int64_t col = cbase + 4 * c4;
                        // N % 8 == 0: a 4-column group is all in or all out
                        if (4 * c4 < ncols && col < args.N)
                            *reinterpret_cast<int4*>(dst + col) =
                                make_int4(run[4 * c4], run[4 * c4 + 1], run[4 * c4 + 2], run[4 * c4 + 3]);
                    }
                }
            } else {
                using OT = OutType<OUT>;
                constexpr int PC = OT::PER_CHUNK;
                constexpr int BOX = OT::BOX_COLS;
                const int64_t row0 = m0 + quarter * 32;
                // A rolled loop over pairs of boxes: its body is fetched once per tile.  The
                // store loop first runs with cold instruction caches (the bench's L2 flush
                // evicts code too); fully unrolled, that first pass held up the epilogue long
                // enough for both accumulators to fill and the MMAs to stall.  Each pass
                // converts run[0 .. 2 BOX) and shifts the sums down by 2 BOX, so indices stay
                // compile-time (one shift per two boxes: 0.5-1% faster than one per box).
#pragma unroll 1
                for (int g2 = 0; g2 < 128 / BOX; g2 += 2) {
                  bool stop = false;
#pragma unroll
                  for (int h = 0; h < 2; ++h) {  // two boxes per pass: run[h * BOX ..]
                    const int g = g2 + h;
                    const int64_t col0 = cbase + g * OT::BOX_COLS;
                    if (g * OT::BOX_COLS >= ncols || col0 >= args.N || row0 >= args.M) {
                        stop = true;  // warp-uniform: nothing of this box is inside the tile and y
                        break;
                    }
                    uint8_t* buf = obuf + (nstore & 1u) * OUT_BUF_BYTES;
                    if (lane == 0)
                        bulk_wait_group_read<1>();  // the store that last used `buf` has read it
                    __syncwarp();
#pragma unroll
                    for (int c = 0; c < 4; ++c) {  // one 16-byte chunk of the row: PC columns
                        const int j0 = h * BOX + c * PC;  // first running sum of the chunk (after the shifts)
                        const int64_t col = col0 + c * PC;
                        // the columns' w_scale and bias from the lanes that loaded them (columns
                        // past N hold 0: computed, then clipped by the store)
                        float wsv[PC], bv[PC];
                        const int src = (g * OT::BOX_COLS + c * PC) >> 2;
#pragma unroll
                        for (int i = 0; i < PC; ++i) {
                            wsv[i] = args.scalar_scales ? ws_scalar : __shfl_sync(0xffffffffu, wsr[i & 3], src + (i >> 2));
                            bv[i] = __shfl_sync(0xffffffffu, bsr[i & 3], src + (i >> 2));
                        }
                        // this lane's residual: 16 bytes of its own row (the element it writes)
                        float rv[PC];
                        if (RES && row < args.M && col < args.N) {
                            const uint4 rr = __ldcg(reinterpret_cast<const uint4*>(
                                static_cast<const uint8_t*>(args.residual) + (row * args.N + col) * OT::BYTES));
                            unpack_out<OUT>(rr, rv);
                        } else {
#pragma unroll
                            for (int i = 0; i < PC; ++i)
                                rv[i] = 0.0f;
                        }
                        // two columns per packed fp32x2 instruction, each lane rounded like the
                        // scalar __fmul_rn / __fadd_rn, in the same order.  The adds are
                        // fma(u, one, v): a packed add taking a packed product with no other use
                        // was fused into one fma by the compiler (CUDA 13.0, sm_103a: despite .rn
                        // and -fmad=false), which rounds once where the layer rounds twice; an
                        // fma by a 1.0 the compiler cannot see is exactly the add, never fused.
                        const float2 one2 = make_float2(args.one, args.one);
                        float t[PC];
#pragma unroll
                        for (int i = 0; i < PC; i += 2) {
                            float2 u;
                            if (MIXED) {  // 16-bit activations: (sum * w_scale) + bias
                                u = make_float2(__int_as_float(run[j0 + i]), __int_as_float(run[j0 + i + 1]));
                            } else {
                                u = make_float2(__int2float_rn(run[j0 + i]), __int2float_rn(run[j0 + i + 1]));
                                u = f2_mul_rn(u, make_float2(xsv, xsv));
                            }
                            u = f2_mul_rn(u, make_float2(wsv[i], wsv[i + 1]));
                            if (args.bias)
                                u = f2_fma_rn(u, one2, make_float2(bv[i], bv[i + 1]));
                            if (RES)
                                u = f2_fma_rn(u, one2, make_float2(rv[i], rv[i + 1]));
                            t[i] = u.x;
                            t[i + 1] = u.y;
                        }
                        uint32_t packed[4];
                        if (OUT == kOutF32) {
#pragma unroll
                            for (int i = 0; i < 4; ++i)
                                packed[i] = __float_as_uint(t[i]);
                        } else {
#pragma unroll
                            for (int i = 0; i < 4; ++i)
                                packed[i] = pack2<OUT>(t[2 * i], t[2 * i + 1]);
                        }
                        // 64-byte swizzle: 16-byte chunk c of row r lives at chunk c ^ ((r >> 1) & 3)
                        const uint32_t phys = (uint32_t)c ^ (((uint32_t)lane >> 1) & 3u);
                        *reinterpret_cast<uint4*>(buf + lane * OUT_ROW_BYTES + phys * 16) =
                            make_uint4(packed[0], packed[1], packed[2], packed[3]);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&tmY, buf, (int32_t)col0, (int32_t)row0);
                        bulk_commit_group();
                    }
                    ++nstore;
                  }
                  if (stop)
                      break;
#pragma unroll
                  for (int j = 0; j < 128 - 2 * BOX; ++j)
                      run[j] = run[j + 2 * BOX];
                }
            }
        }
        // the stores must have read shared memory before it is released; their writes to
        // global memory complete with the grid
        if (lane == 0)
            bulk_wait_group_read<0>();
        __syncwarp();
    }

    griddep_launch_dependents();
    tc_fence_before();
    // every warp is converged here: all TMEM reads of this CTA are done and, in a pair,
    // the leader's MMAs (which write this CTA's TMEM and read its shared memory) as well
    if (PAIR)
        cluster_sync();
    else
        __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        if (PAIR)
            tmem_dealloc_pair(tmem_base, TMEM_COLS);
        else
            tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

// The self-test of the bounded wait: one thread waits on a barrier that expects one
// arrival that never comes.
__global__ void wait_selftest_kernel(uint64_t timeout_ns)
{
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0)
        mbar_wait(&bar, 0, &abort_flag, &g_device_error, kErrWaitSelfTest, timeout_ns);
}

}  // namespace gemm

// ---------------------------------------------------------------- host side
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// 2-D row-major tensor of `rows` x `cols` elements with a row pitch of `pitch_bytes`;
// false (with a message in *why) when the driver rejects it.
static bool make_map_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t cols, uint64_t rows,
                 uint64_t pitch_bytes, uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle swz, std::string* why)
{
    auto fn = encode_fn();
    if (!fn) {
        *why = "cuTensorMapEncodeTiled is not available from the driver";
        return false;
    }
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {pitch_bytes};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        char msg[160];
        snprintf(msg, sizeof msg, "cuTensorMapEncodeTiled failed (%d) for a %llux%llu tensor", (int)r,
                 (unsigned long long)rows, (unsigned long long)cols);
        *why = msg;
        return false;
    }
    return true;
}

template <bool RAW, bool PAIR, int OUT, bool MIXED, bool SPLIT, bool RES>
static cudaError_t ensure_smem_attr(int device)
{
    (void)device;
    // a kernel attribute belongs to the context it was set in: set once per context
    static ContextCache<int> cache;
    int done = 0;
    return cache.get(&done, [](int* d) {
        cudaError_t e = cudaFuncSetAttribute(gemm::gemm_kernel<RAW, PAIR, OUT, MIXED, SPLIT, RES>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)gemm::Mode<PAIR>::SMEM_BYTES);
        if (e == cudaSuccess) {
            // the warpgroups' register re-balancing must fit in what a block is launched
            // with (registers are granted per warp in units of 8 per thread), else the
            // epilogue's increase would wait forever: refuse to launch instead
            cudaFuncAttributes fa;
            e = cudaFuncGetAttributes(&fa, gemm::gemm_kernel<RAW, PAIR, OUT, MIXED, SPLIT, RES>);
            if (e == cudaSuccess &&
                (uint64_t)((fa.numRegs + 7) / 8 * 8) * gemm::THREADS < (uint64_t)gemm::REGS_NEEDED_PER_BLOCK)
                e = cudaErrorInvalidConfiguration;
        }
        *d = 1;
        return e;
    });
}

static cudaLaunchConfig_t make_config(bool pair, size_t smem, cudaStream_t s, cudaLaunchAttribute (&attr)[2])
{
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(gemm::THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = pair ? 2 : 1;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pair ? 2 : 1;
    return cfg;
}

// How many units (pairs, or single CTAs) can be resident at once: a pair needs two SMs
// of one GPC, so for pairs the count comes from the occupancy calculator.
template <bool PAIR>
static cudaError_t resident_units(const DeviceInfo& dev, int64_t* out)
{
    if (!PAIR) {
        *out = dev.sm_count;
        return cudaSuccess;
    }
    static int cached[64] = {};
    static std::mutex mu;
    std::lock_guard<std::mutex> lock(mu);
    int& n = cached[(dev.device >= 0 && dev.device < 64) ? dev.device : 0];
    if (n == 0) {
        cudaError_t e = ensure_smem_attr<false, true, gemm::kOutBf16, false, false, false>(dev.device);
        if (e != cudaSuccess)
            return e;
        cudaLaunchAttribute attr[2];
        cudaLaunchConfig_t cfg = make_config(true, gemm::Mode<true>::SMEM_BYTES, nullptr, attr);
        cfg.gridDim = dim3(2 * (dev.sm_count / 2));
        e = cudaOccupancyMaxActiveClusters(&n, gemm::gemm_kernel<false, true, gemm::kOutBf16, false, false, false>,
                                           &cfg);
        if (e != cudaSuccess)
            return e;
        if (n <= 0)
            return cudaErrorInvalidConfiguration;
    }
    *out = n;
    return cudaSuccess;
}

// Time of 64 deep of K of one unit, in units of 0.01 ns, as measured on GB300 over tile
// widths 32..256 (25900x16384x4096, many waves): a CTA pair's 256-row unit (128-deep
// stages) takes about 218 + 0.41 * bn ns, a single CTA's 128-row unit (64-deep stages)
// about 295 + 0.35 * bn ns.  Narrow tiles save little per k-block, so the width mainly
// trades wave quantization.
static int64_t kblock_cost(bool pair, int bn)
{
    return pair ? 21800 + 41 * (int64_t)bn : 29500 + 35 * (int64_t)bn;
}

// A launch of CTA pairs costs about 2 us more than one of single CTAs (2-CTA cluster
// launch and set-up, the pair's longer last epilogue): measured on a one-wave problem
// (1024x4096x4096) as the launch time minus the k-block costs above, per mode.  The
// term only decides problems of one or two waves.
constexpr int64_t kPairLaunchCost = 210000;

// A K-split tail slice must keep at least this many k-blocks.  Publishing the slices'
// sums (write, fence, count the arrival) and adding them in the last slice cost, as
// measured on GB300 (2-, 3- and 4-way splits of 64- and 48-k-block units), about
// kSplitFixedKb + kSplitPerSliceKb * split k-block times.
constexpr int kMinSliceKb = 4;
constexpr int64_t kSplitFixedKb = 10;
constexpr int64_t kSplitPerSliceKb = 10;

// Cost of one configuration: `units` run as waves of `resident`; the last partial wave,
// if any, either runs whole or is split `split` ways along K over the idle units.
struct TileCost {
    int64_t cost;
    int split;
    int64_t full_units;
};

static TileCost tile_cost(bool pair, int bn, int64_t units, int64_t resident, int num_kb, int64_t tail_ctas,
                          int force_split)
{
    const int64_t waves = units / resident, tail = units % resident;
    TileCost c{(waves + (tail ? 1 : 0)) * num_kb, 1, units};
    if (tail && force_split != 1) {
        const int64_t ranks = pair ? 2 : 1;
        const int64_t smax = std::min(std::min(resident / tail, (int64_t)(num_kb / kMinSliceKb)),
                                      std::min((int64_t)kTailMaxSplit, tail_ctas / (tail * ranks)));
        for (int sp = 2; sp <= smax; ++sp) {
            if (force_split > 1 && sp != force_split)
                continue;
            const int64_t kbs = waves * num_kb + (num_kb + sp - 1) / sp + kSplitFixedKb + kSplitPerSliceKb * sp;
            if (kbs < c.cost || force_split > 1) {
                c.cost = kbs;
                c.split = sp;
                c.full_units = waves * resident;
            }
        }
    }
    c.cost = c.cost * kblock_cost(pair, bn) + (pair ? kPairLaunchCost : 0);
    return c;
}

// The configuration that finishes soonest.  CK_GEMM_BN=<width> forces a width,
// CK_GEMM_SPLIT=1 turns the K-split tail off and CK_GEMM_SPLIT=<s> asks for s slices
// where the tail allows it (A/B timing).
static void choose_tile(int64_t M, int64_t N, int num_kb, int64_t tiles_m, int64_t resident_pair,
                        int64_t resident_single, bool pair_allowed, bool single_allowed, bool no_split,
                        GemmPlan* plan)
{
    int force_bn = 0, force_split = 0;
    if (const char* f = std::getenv("CK_GEMM_BN")) {
        const int v = std::atoi(f);
        if (v >= 32 && v <= gemm::BN && v % 32 == 0)
            force_bn = v;
    }
    if (const char* f = std::getenv("CK_GEMM_SPLIT")) {
        const int v = std::atoi(f);
        if (v >= 1 && v <= kTailMaxSplit)
            force_split = v;
    }
    if (no_split)
        force_split = 1;
    const int64_t tail_ctas = gemm_tail_ctas(M, N);
    int64_t best_cost = -1;
    bool best_forced = false;  // the best so far has the requested split
    for (int p = pair_allowed ? 1 : 0; p >= (single_allowed ? 0 : 1); --p) {
        const int64_t units_m = p ? (tiles_m + 1) / 2 : tiles_m;
        const int64_t resident = p ? resident_pair : resident_single;
        for (int bn = gemm::BN; bn >= 32; bn -= 32) {
            if (force_bn && bn != force_bn)
                continue;
            const int64_t units = units_m * ((N + bn - 1) / bn);
            const TileCost c = tile_cost(p != 0, bn, units, resident, num_kb, tail_ctas, force_split);
            // a requested split wins over cheaper configurations that cannot have it
            const bool forced = force_split > 1 && c.split == force_split;
            if (best_forced && !forced)
                continue;
            if (best_cost < 0 || c.cost < best_cost || (forced && !best_forced)) {
                best_forced = forced;
                best_cost = c.cost;
                plan->pair = p != 0;
                plan->bn = bn;
                plan->resident = resident;
                plan->units = units;
                plan->full_units = c.full_units;
                plan->split = c.split;
            }
        }
    }
}

// Launch with programmatic stream serialization and, for pairs, 2-CTA clusters; the
// persistent grid is as many units as can be resident at once.
template <bool RAW, bool PAIR, int OUT, bool MIXED, bool SPLIT, bool RES>
static cudaError_t launch_kernel(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmY,
                                 const gemm::Args& a, const DeviceInfo& dev, cudaStream_t s)
{
    using namespace gemm;
    cudaError_t e = ensure_smem_attr<RAW, PAIR, OUT, MIXED, SPLIT, RES>(dev.device);
    if (e != cudaSuccess)
        return e;
    int64_t resident = 0;
    if ((e = resident_units<PAIR>(dev, &resident)) != cudaSuccess)
        return e;
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = make_config(PAIR, Mode<PAIR>::SMEM_BYTES, s, attr);
    const int64_t units = std::min<int64_t>(a.num_items, resident);
    cfg.gridDim = dim3((unsigned)(PAIR ? 2 * units : units));
    return cudaLaunchKernelEx(&cfg, gemm_kernel<RAW, PAIR, OUT, MIXED, SPLIT, RES>, tmA, tmB, tmY, a);
}

// A 64-bit tag no earlier launch of this process used (high-entropy start, so slots
// left in recycled memory by another process do not match either); never 0.
static unsigned long long next_gemm_epoch()
{
    static std::atomic<unsigned long long> counter([] {
        unsigned long long z = (unsigned long long)std::chrono::steady_clock::now().time_since_epoch().count() ^
                               ((unsigned long long)getpid() << 31) ^ 0xD1B54A32D192ED03ull;
        z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;  // splitmix64 finaliser
        z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
        return z ^ (z >> 31);
    }());
    unsigned long long e;
    do {
        e = counter.fetch_add(1, std::memory_order_relaxed);
    } while (e == 0);
    return e;
}

cudaError_t plan_gemm(int64_t M, int64_t N, int64_t K, bool mixed, const DeviceInfo& dev, GemmPlan* plan)
{
    const int64_t tiles_m = (M + gemm::BM - 1) / gemm::BM;
    // CK_GEMM_PAIR=0 / =1 restricts the choice to single CTAs / CTA pairs (A/B timing);
    // a problem with one 128-row tile row always runs single CTAs
    const char* force = std::getenv("CK_GEMM_PAIR");
    const bool pair_allowed = tiles_m >= 2 && !(force && std::strcmp(force, "0") == 0);
    const bool single_allowed = !(pair_allowed && force && std::strcmp(force, "1") == 0);
    int64_t resident_pair = 0, resident_single = 0;
    cudaError_t e = resident_units<false>(dev, &resident_single);
    if (e == cudaSuccess && pair_allowed)
        e = resident_units<true>(dev, &resident_pair);
    if (e != cudaSuccess)
        return e;
    const int num_kb = (int)((K + gemm::BK - 1) / gemm::BK);
    // the 16-bit-activation kernels keep one fp32 sum per tile: no K-split
    choose_tile(M, N, num_kb, tiles_m, resident_pair, resident_single, pair_allowed, single_allowed, mixed, plan);
    return cudaSuccess;
}

std::string describe_gemm_plan(int64_t M, int64_t N, int64_t K, bool mixed, bool split_allowed,
                               const DeviceInfo& dev)
{
    GemmPlan plan;
    if (plan_gemm(std::max<int64_t>(M, 1), N, K, mixed, dev, &plan) != cudaSuccess)
        return "no GEMM plan (device query failed)";
    char buf[192];
    const int split = split_allowed ? plan.split : 1;
    snprintf(buf, sizeof buf, "%d-wide tiles on %s (%lld units, %lld resident)%s", plan.bn,
             plan.pair ? "CTA pairs of 256 rows" : "single CTAs of 128 rows", (long long)plan.units,
             (long long)plan.resident, split > 1 ? ", last wave split along K" : "");
    std::string r = buf;
    if (split > 1)
        r += " " + std::to_string(split) + " ways";
    return r;
}

// The dequant kernels by output type, tile mode, K-split and residual.
template <bool MIXED, bool SPLIT, bool RES>
static cudaError_t launch_dequant(bool pair, int out_dtype, const CUtensorMap& tmA, const CUtensorMap& tmB,
                                  const CUtensorMap& tmY, const gemm::Args& a, const DeviceInfo& dev,
                                  cudaStream_t s)
{
    using namespace gemm;
    switch (out_dtype) {
    case kOutF16:
        return pair ? launch_kernel<false, true, kOutF16, MIXED, SPLIT, RES>(tmA, tmB, tmY, a, dev, s)
                    : launch_kernel<false, false, kOutF16, MIXED, SPLIT, RES>(tmA, tmB, tmY, a, dev, s);
    case kOutF32:
        return pair ? launch_kernel<false, true, kOutF32, MIXED, SPLIT, RES>(tmA, tmB, tmY, a, dev, s)
                    : launch_kernel<false, false, kOutF32, MIXED, SPLIT, RES>(tmA, tmB, tmY, a, dev, s);
    default:
        return pair ? launch_kernel<false, true, kOutBf16, MIXED, SPLIT, RES>(tmA, tmB, tmY, a, dev, s)
                    : launch_kernel<false, false, kOutBf16, MIXED, SPLIT, RES>(tmA, tmB, tmY, a, dev, s);
    }
}

template <bool MIXED, bool SPLIT>
static cudaError_t launch_dequant(bool res, bool pair, int out_dtype, const CUtensorMap& tmA,
                                  const CUtensorMap& tmB, const CUtensorMap& tmY, const gemm::Args& a,
                                  const DeviceInfo& dev, cudaStream_t s)
{
    return res ? launch_dequant<MIXED, SPLIT, true>(pair, out_dtype, tmA, tmB, tmY, a, dev, s)
               : launch_dequant<MIXED, SPLIT, false>(pair, out_dtype, tmA, tmB, tmY, a, dev, s);
}

cudaError_t launch_gemm(const GemmProblem& p, const DeviceInfo& dev, cudaStream_t s, std::string* why)
{
    using namespace gemm;
    const bool raw = p.acc != nullptr;
    CUtensorMap tmA, tmB, tmY;
    if (!make_map_2d(&tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.a, p.K, p.M, (uint64_t)p.K * 2, BK, BM,
                     CU_TENSOR_MAP_SWIZZLE_128B, why))
        return cudaErrorInvalidValue;
    if (!raw && p.out_dtype != kOutBf16 && p.out_dtype != kOutF16 && p.out_dtype != kOutF32) {
        *why = "unknown output type";
        return cudaErrorInvalidValue;
    }
    if (raw) {
        tmY = tmA;  // unused by the raw-accumulator kernel
    } else {
        const bool f32 = p.out_dtype == kOutF32;
        const CUtensorMapDataType dt = f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                           : (p.out_dtype == kOutF16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                                     : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16);
        const uint32_t esize = f32 ? 4u : 2u;
        if (!make_map_2d(&tmY, dt, p.y, p.N, p.M, (uint64_t)p.N * esize, OUT_ROW_BYTES / esize, 32,
                         CU_TENSOR_MAP_SWIZZLE_64B, why))
            return cudaErrorInvalidValue;
    }
    Args a;
    a.M = p.M;
    a.N = p.N;
    a.K = p.K;
    a.xs = p.x_scale;
    a.ws = p.w_scale;
    a.bias = reinterpret_cast<const __nv_bfloat16*>(p.bias);
    a.residual = p.residual;
    a.acc = p.acc;
    a.tiles_m = (int)((p.M + BM - 1) / BM);
    a.scalar_scales = p.scalar_scales;
    a.timeout_ns = DEFAULT_TIMEOUT_NS;
    a.one = 1.0f;
    GemmPlan plan;
    const cudaError_t e = plan_gemm(p.M, p.N, p.K, p.mixed, dev, &plan);
    if (e != cudaSuccess)
        return e;
    const bool pair = plan.pair;
    a.unit_rows = pair ? 2 : 1;
    a.units_m = (a.tiles_m + a.unit_rows - 1) / a.unit_rows;
    // Grouped order: the resident units sweep N together over a band of tile rows.  When
    // both operands fit in L2 together (up to 80 MB of bf16 codes) a 1024-row band is
    // best; larger problems take a band of about 32 MB of activation rows (1024 to 4096
    // rows), which stays in L2 while the weight streams past it, so the weight is read
    // from HBM about once per band.  Measured on GB300 (interleaved runs), a 24 MB band
    // against the 1024-row one: 4096x12288x3072 0.180 -> 0.168 ms, 8192x16384x4096 0.579 ->
    // 0.541, 25900x16384x4096 1.869 -> 1.772, 80666x28672x5376 13.95 -> 13.52,
    // 99865x21504x5376 12.66 -> 12.24 (4096^3 was 3.7% slower with the wider band and keeps
    // 1024 rows); 32 MB against 24 MB, GEMM launches under the power cap: 80666x28672x5376
    // 13.39 -> 13.20 ms, 99865x21504x5376 12.51 -> 12.24, 8192x16384x4096 0.531 -> 0.530,
    // 25900x16384x4096 1.74 -> 1.73; wider bands lose the weight's reuse in L2 (80666x28672x5376:
    // 38 MB 13.23 ms, 50 MB 13.55, 66 MB 14.3).
    // CK_GEMM_GROUP=<units per band> overrides (A/B timing).
    const bool fits_l2 = 2 * p.K * (p.M + p.N) <= ((int64_t)80 << 20);
    const int64_t band_rows =
        fits_l2 ? 1024 : std::min<int64_t>(4096, std::max<int64_t>(1024, ((int64_t)32 << 20) / (2 * p.K)));
    a.group_m = (int)std::max<int64_t>(1, band_rows / (pair ? 2 * BM : BM));
    if (const char* g = std::getenv("CK_GEMM_GROUP")) {  // unit rows per sweep over N (A/B timing)
        const int v = std::atoi(g);
        if (v >= 1 && v <= 4096)
            a.group_m = v;
    }
    a.bn = plan.bn;
    a.tiles_n = (int)((p.N + a.bn - 1) / a.bn);
    a.num_units = (int64_t)a.units_m * a.tiles_n;
    a.split = 1;
    a.full_units = a.num_units;
    a.num_items = a.num_units;
    a.partials = nullptr;
    a.tail_slots = nullptr;
    a.epoch = 0;
    if (plan.split > 1 && p.tail != nullptr && plan.units == a.num_units) {
        const int64_t ctas = gemm_tail_ctas(p.M, p.N);
        a.split = plan.split;
        a.full_units = plan.full_units;
        a.num_items = a.full_units + (a.num_units - a.full_units) * a.split;
        a.partials = static_cast<int32_t*>(p.tail);
        a.tail_slots = reinterpret_cast<unsigned long long*>(static_cast<uint8_t*>(p.tail) + ctas * kTailCtaBytes);
        a.epoch = next_gemm_epoch();
    }
    a.idesc = (pair ? Mode<true>::IDESC_M : Mode<false>::IDESC_M) | ((uint32_t)(a.bn >> 3) << 17);
    const int kb_depth = pair ? Mode<true>::KB : Mode<false>::KB;  // K per k-block of this mode
    a.num_kb = (int)((p.K + kb_depth - 1) / kb_depth);
    a.chunk_kb = p.mixed ? a.num_kb : CHUNK_K / kb_depth;
    a.tx_bytes = (pair ? 2u : 1u) * (uint32_t)(kb_depth / BK) * (A_BYTES + (uint32_t)(pair ? a.bn / 2 : a.bn) * BK * 2);
    if (!make_map_2d(&tmB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.b, p.K, p.N, (uint64_t)p.K * 2, BK, a.bn / 2,
                     CU_TENSOR_MAP_SWIZZLE_128B, why))
        return cudaErrorInvalidValue;
    const bool split = a.split > 1;  // never for the 16-bit path (planned without)
    if (raw) {
        if (split)
            return pair ? launch_kernel<true, true, kOutBf16, false, true, false>(tmA, tmB, tmY, a, dev, s)
                        : launch_kernel<true, false, kOutBf16, false, true, false>(tmA, tmB, tmY, a, dev, s);
        return pair ? launch_kernel<true, true, kOutBf16, false, false, false>(tmA, tmB, tmY, a, dev, s)
                    : launch_kernel<true, false, kOutBf16, false, false, false>(tmA, tmB, tmY, a, dev, s);
    }
    const bool res = p.residual != nullptr;
    if (p.mixed)
        return launch_dequant<true, false>(res, pair, p.out_dtype, tmA, tmB, tmY, a, dev, s);
    if (split)
        return launch_dequant<false, true>(res, pair, p.out_dtype, tmA, tmB, tmY, a, dev, s);
    return launch_dequant<false, false>(res, pair, p.out_dtype, tmA, tmB, tmY, a, dev, s);
}

cudaError_t read_device_error(unsigned int* value, bool clear)
{
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess)
        return e;
    e = cudaMemcpyFromSymbol(value, g_device_error, sizeof(unsigned int));
    if (e != cudaSuccess || !clear)
        return e;
    const unsigned int zero = 0;
    return cudaMemcpyToSymbol(g_device_error, &zero, sizeof zero);
}

cudaError_t device_error_ptr(unsigned int** ptr)
{
    static ContextCache<unsigned int*> cache;
    return cache.get(ptr, [](unsigned int** p) {
        void* a = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&a, g_device_error);
        *p = static_cast<unsigned int*>(a);
        return e;
    });
}

cudaError_t launch_wait_selftest(uint64_t timeout_ns, cudaStream_t s)
{
    gemm::wait_selftest_kernel<<<1, 32, 0, s>>>(timeout_ns);
    return cudaGetLastError();
}

}  // namespace ck
