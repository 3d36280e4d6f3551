// Fused SSD forward on tcgen05: all four steps of "Accelerating Mamba-2 with
// High-Performance Forward Pass Kernels in NVIDIA CUDA Tile" (the in-chunk
// cumulative sum, the per-chunk state and its sequential pass, and
// compute_out) in one kernel, so x is read once, y written once and no
// intermediate reaches HBM.
//
// One CTA walks one (batch, head) slab -- or one segment of it -- in blocks
// of 128 tokens.  A chunk of Q = 128 k tokens is evaluated as k such blocks:
// its off-diagonal decay blocks are applied through the state at the block
// boundary, by associativity,
//     (C_1 B_0^T o decay) (dt x_0) = 2^(g_1) C_1 (B_0^T (w o x_0)),
// the same product in a different order.  Per block, with g the block-local
// cumulative sum of A dt (log2 units):
//     CB    = C B^T                                  tensor cores -> TMEM
//     S^T   = B^T (w o x),  w_j = 2^(g_end - g_j) dt_j   tensor cores -> TMEM
//     L_ij  = [j <= i] CB_ij 2^(g_i - g_j) dt_j + [i = j] D
//                                                    math warps, in place in TMEM (bf16)
//     intra = L x                                    tensor cores, A read from TMEM
//     inter = C h^T                                  tensor cores -> TMEM
//     y     = 2^(g_i) inter + intra                  math warps (drain)
//     h     = 2^(g_end) h + S                        math warps, fp32 in registers
// dt_j is folded into the exponent, 2^(g_i - g_j + log2 dt_j) (dt_j = 0 gives
// 2^-inf = 0), and the causal selection replaces the exponent of masked
// entries by -inf before it is evaluated, so no positive exponent of the
// decay is ever computed.  The skip term D x rides on the diagonal of L.
//
// Only h(k + 1) = 2^(g_end) h(k) + S(k) is serial, and S(k) does not depend
// on h, so every other product of a block is taken off that chain: S^T is
// issued as soon as w o x is ready, and the state update, the decay operand
// and the y drain each have warps of their own.  The bf16 copy of the state
// that C h^T reads has one buffer: the update of block k writes it once
// C h^T(k) has read it.  Blocks are software-pipelined across two stages of
// the C, B and tensor-memory buffers.
// Roles: warp 0 = TMA producer and the block's cumulative sum (published once
// for every role), warp 1 = tensor-memory owner and MMA issuer, warps 2..7 =
// warpgroup A (the decay operand L), warps 8..11 = warpgroup S (w o x and the
// state), warps 12..15 = warpgroup Y (y and its TMA store).  A math thread
// owns tile row / state row r = its TMEM lane.  One CTA per SM (all 512 TMEM
// columns, 216.4 KiB of shared memory).
#include "ptx_sm100.cuh"
#include "ssd_block_math.cuh"
#define SSD_DBG_FILE 1u   // kDbgFused
#include "ssd_debug.cuh"
#include "ssd_internal.h"
#include "ssd_tc.cuh"
#include "ssd_tmap.h"

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdlib>

namespace ssd {
namespace {


// Work units.  Slabs (batch, head) are numbered heads fastest.  Slabs
// [0, n_whole) are one unit each, walked over the whole sequence; each later
// ("tail") slab is split into nseg segments of seg_len tokens (a multiple of
// 128; the last one may be shorter), one unit each, so the last partial wave
// of slabs spreads over more SMs.  A tail segment s > 0 starts from the state
// seg_hin[tail slab][s] (computed beforehand by the states-only pass and
// the combine kernel).  In the states-only pass (kMode 2) the units
// are segments 0 .. nseg - 2 of every tail slab, started from zero: only
// B^T (w o x) and the state update run, and each unit writes its final state
// to seg_state and the sum of its blocks' log2 decays to seg_decay.
struct FusedParams {
    int64_t L;            // sequence length
    int64_t seg_len;      // tokens per tail segment (multiple of 128)
    int B, H, hpg, nseg;
    const float *dt;
    int64_t dt_sb, dt_sl;
    const float *A;
    const float *D;       // may be null
    const float *h0;      // [B][H][P][N] initial state, or null (= 0)
    float *h_final;       // [B][H][P][N] final state, or null
    __nv_bfloat16 *y;
    int64_t y_sb, y_sl, y_sh;
    unsigned int *err;
    int64_t n_dt, n_hs;   // element extents of dt and of h0 / h_final (debug build)
};

// What only a split launch reads (kept apart so the whole-slab kernel's
// parameters stay as small as they can).
struct SplitParams {
    const float *seg_hin; // [tail slabs][nseg][P][N] entering state of tail segments
    float *seg_state;     // [tail slabs][nseg - 1][P][N] (states-only pass)
    float *seg_decay;     // [tail slabs][nseg - 1]        (states-only pass)
    int n_whole;
    int64_t n_seg_state, n_seg_decay, n_seg_hin;   // element extents (debug build)
};

// Shared memory: the operand tiles first (the 128-byte swizzle pattern repeats
// every 1024 bytes, so they need a 1024-byte aligned base), then small arrays
// and the barriers.
struct FusedSmem {
    static constexpr int kC = 0;          // 2 stages x 2 x [128 tokens][128 B]  C, K-major
    static constexpr int kB = 65536;      // 2 stages x 2 x [128 tokens][128 B]  B, K-major
    static constexpr int kX = 131072;     // 3 slots x [128 tokens][128 B]       x, then y
    static constexpr int kXP = 180224;    // [128 tokens][128 B]                 w o x
    static constexpr int kHB = 196608;    // [128 n][128 B]                      bf16 state
    static constexpr int kF = 212992;     // 4 records: g, ngd, vcol [128]; gpiv [4]; g_end
    static constexpr int kNF = 4 * 392;   // four records (see kRec)
    static constexpr int kDT = kF + kNF * 4;   // [4][128] dt of the next records
    static constexpr int kBar = kDT + 4 * 128 * 4;
    static constexpr int kNBar = 33;
    static constexpr int kBytes = kBar + kNBar * 8 + 8;
};
static_assert(FusedSmem::kBytes <= 232448, "shared memory above the per-CTA limit");

constexpr int kThreads = 512;             // 16 warps: four per scheduler, 128 registers each
constexpr int kWgA = 192;                 // warpgroup A threads (warps 2..7)
// floats of one block's cumulative-sum record (389 used), a multiple of 4 so
// that both records' arrays stay 16-byte aligned for vector loads
constexpr int kRec = 392;
constexpr int kNRec = 4;                  // records in the ring
// warps that read a record: warpgroups A (6), S (4) and Y (4); each releases it once
constexpr int kRecReaders = 14;
static_assert(kRec % 4 == 0 && FusedSmem::kNF == kNRec * kRec && FusedSmem::kF % 16 == 0,
              "record layout");


// Named barriers (0 is __syncthreads): 4 + q = the two warps of warpgroup A
// on TMEM lane quarter q (q = 2, 3), 9 = warpgroup Y, 11 = warpgroup S (the
// states-only pass).
//
// Block k uses stage s = k & 1 of the double buffers.  Tensor memory:
// [128 s, +128) = C B^T, then L in its first 64 columns and the intra
// accumulator in its last 64; [256 + 64 s, +64) = S^T; [384 + 64 s, +64) =
// inter.  x(k) lands in slot k mod 3 of a three-slot pool, where y(k) is
// staged once L x(k) has read x(k); the slot is reloaded once the TMA store
// of y(k) has read it.  w o x and the bf16 state operand have one buffer
// each: w o x(k + 1) is written once B^T (w o x)(k) has completed, the state
// entering block k + 1 once C h^T(k) has read the one entering block k.
//
// Every wait below names the phase of a barrier that cannot have advanced a
// further phase yet: the later phase depends on work that the waiter itself
// enables.
// kMode: 0 = every unit a whole slab, 1 = whole slabs then tail segments,
// 2 = the states-only pass over tail segments.  The unit is blockIdx.x.
template <int kMode>
__device__ __forceinline__ void unit_range(const FusedParams &p, const SplitParams &sp,
                                           size_t &slab, int64_t &t_begin, int64_t &t_end) {
    const int unit = blockIdx.x;
    int sg = 0;
    if (kMode == 1 && unit < sp.n_whole) {
        slab = size_t(unit);
        t_begin = 0;
        t_end = p.L;
        return;
    }
    if (kMode == 2) {
        slab = size_t(sp.n_whole) + unit / (p.nseg - 1);
        sg = unit % (p.nseg - 1);
    } else {
        slab = size_t(sp.n_whole) + (unit - sp.n_whole) / p.nseg;
        sg = (unit - sp.n_whole) % p.nseg;
    }
    t_begin = int64_t(sg) * p.seg_len;
    t_end = t_begin + p.seg_len < p.L ? t_begin + p.seg_len : p.L;
}

// State entering the unit ([P][N] fp32), or null for zero.
template <int kMode>
__device__ __forceinline__ const float *unit_h_in(const FusedParams &p, const SplitParams &sp,
                                                  size_t slab) {
    constexpr size_t PN = 8192;
    const int unit = blockIdx.x;
    if (kMode == 2) return nullptr;
    if (kMode == 1 && unit >= sp.n_whole && (unit - sp.n_whole) % p.nseg != 0)
        return sp.seg_hin + size_t(unit - sp.n_whole) * PN;
    return p.h0 ? p.h0 + slab * PN : nullptr;
}

// Where the unit's final state goes, or null.
template <int kMode>
__device__ __forceinline__ float *unit_h_out(const FusedParams &p, const SplitParams &sp,
                                             size_t slab) {
    constexpr size_t PN = 8192;
    const int unit = blockIdx.x;
    if (kMode == 2) return sp.seg_state + size_t(unit) * PN;
    if (kMode == 1 && unit >= sp.n_whole && (unit - sp.n_whole) % p.nseg != p.nseg - 1)
        return nullptr;
    return p.h_final ? p.h_final + slab * PN : nullptr;
}

template <int kMode>
__global__ void __launch_bounds__(kThreads, 1)
k_ssd_fused(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_b,
            const __grid_constant__ CUtensorMap tm_c, const __grid_constant__ CUtensorMap tm_y,
            const FusedParams p, const SplitParams sp) {
    using SM = FusedSmem;
    constexpr uint32_t kCols = 512;
    constexpr uint32_t kIdCB = ptx::idesc_bf16_f32(128, 128, false, false);
    constexpr uint32_t kIdKmn = ptx::idesc_bf16_f32(128, 64, false, true);   // A K-major, B MN-major
    constexpr uint32_t kIdMnmn = ptx::idesc_bf16_f32(128, 64, true, true);
    extern __shared__ __align__(1024) uint8_t smem[];
    if (ptx::smem_u32(smem) & 1023u) {   // uniform over the CTA: nothing has started yet
        if (threadIdx.x == 0) atomicOr(p.err, kErrSmemAlign);
        return;
    }
    float *rec_all = reinterpret_cast<float *>(smem + SM::kF);   // [kNRec][kRec]
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + SM::kBar);
    uint64_t *full_C = bars, *full_B = bars + 2, *cb_done = bars + 4, *s_done = bars + 6,
             *inter_done = bars + 8, *intra_done = bars + 10, *L_ready = bars + 12,
             *st_done = bars + 14, *drain_done = bars + 16, *xp_ready = bars + 18,
             *sc_ready = bars + 19, *rec_free = bars + 23, *full_X = bars + 27,
             *xfree = bars + 30;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + SM::kNBar);
    int *s_err = reinterpret_cast<int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr bool states_only = kMode == 2;
    // this unit's slab (heads fastest, so neighbouring CTAs share B, C in L2)
    // and token range; its entering and final states are looked up where
    // they are used, so no pointer stays live through the block loops
    size_t slab;
    int64_t t_begin, t_end;
    int h, b, seg = 0;
    if constexpr (kMode == 0) {
        // every unit a whole slab (seg_len covers the sequence)
        const int unit = blockIdx.x;
        h = unit % p.H;
        b = (unit / p.H) % p.B;
        seg = unit / (p.H * p.B);
        t_begin = int64_t(seg) * p.seg_len;
        t_end = t_begin + p.seg_len < p.L ? t_begin + p.seg_len : p.L;
        slab = size_t(b) * p.H + h;
    } else {
        unit_range<kMode>(p, sp, slab, t_begin, t_end);
        h = int(slab) % p.H;
        b = int(slab) / p.H;
    }
    const int g = h / p.hpg;
    const int nblk = int((t_end - t_begin + 127) / 128);

    if (threadIdx.x == 0) {
        for (int s = 0; s < 2; ++s) {
            ptx::mbar_init(&full_C[s], 1);
            ptx::mbar_init(&full_B[s], 1);
            ptx::mbar_init(&cb_done[s], 1);
            ptx::mbar_init(&s_done[s], 1);
            ptx::mbar_init(&inter_done[s], 1);
            ptx::mbar_init(&intra_done[s], 1);
            ptx::mbar_init(&L_ready[s], kWgA);
            ptx::mbar_init(&st_done[s], 128);
            ptx::mbar_init(&drain_done[s], 128);
        }
        ptx::mbar_init(xp_ready, 128);
        for (int i = 0; i < kNRec; ++i) {
            ptx::mbar_init(&sc_ready[i], 32);
            ptx::mbar_init(&rec_free[i], states_only ? 4 : kRecReaders);
        }
        for (int i = 0; i < 3; ++i) {
            ptx::mbar_init(&full_X[i], 1);
            ptx::mbar_init(&xfree[i], 1);
        }
        *s_err = 0;
        ptx::fence_mbar_init();
        ptx::prefetch_tmap(&tm_x);
        ptx::prefetch_tmap(&tm_b);
        ptx::prefetch_tmap(&tm_c);
        ptx::prefetch_tmap(&tm_y);
    }
    if (warp == 1) {
        ptx::tmem_alloc(tmem_slot, kCols);
        ptx::tmem_relinquish();
    }
    // warpgroup S: the entering state, fp32 in registers and bf16 in operand buffer 0
    float2 hreg[32];   // state row n = r, headdim pairs (2m, 2m + 1)
    if (warp >= 8 && warp < 12) {
        const int r = 32 * (warp & 3) + lane;
        const float *hin;
        if constexpr (kMode == 0)
            hin = p.h0 ? p.h0 + (size_t(seg) * p.B * p.H + slab) * 8192 : nullptr;
        else
            hin = unit_h_in<kMode>(p, sp, slab);
        if (hin) {   // the debug build checks the slab's span
            const bool from_seg = kMode != 0 && sp.seg_hin && hin >= sp.seg_hin &&
                                  hin < sp.seg_hin + sp.n_seg_hin;
            if (from_seg ? !SSD_SPAN_OK(p.err, hin, sp.seg_hin, sp.n_seg_hin, 8192)
                         : !SSD_SPAN_OK(p.err, hin, p.h0, p.n_hs, 8192))
                hin = nullptr;
        }
#pragma unroll
        for (int m = 0; m < 32; ++m)
            hreg[m] = hin ? make_float2(hin[(2 * m) * 128 + r], hin[(2 * m + 1) * 128 + r])
                          : make_float2(0.f, 0.f);
        write_state_row(smem + SM::kHB, r, hreg);
        ptx::fence_proxy_async_smem();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    bool ok = true;

    if (warp == 0) {
        // ---------------- TMA producer and the cumulative-sum record ----------------
        const float Ah = SSD_IDX_OK(p.err, h, p.H) ? p.A[h] : 0.f;
        const float *dtp = p.dt + int64_t(b) * p.dt_sb + h;
        // Event loop, warp-uniform: lane 0 tests the barriers and issues the
        // copies, the whole warp builds the records.  Each stream goes ahead as
        // soon as its own buffer is free, so no copy waits behind another.
        // dt of record j is copied asynchronously into ring slot j & 3, four
        // records ahead; each lane copies, and later reads, its own four rows.
        float *dtring = reinterpret_cast<float *>(smem + SM::kDT);
        auto fetch_dt = [&](int j) {
            float *dst = dtring + 128 * (j & 3);
#pragma unroll
            for (int qq = 0; qq < 4; ++qq) {
                const int row = 32 * qq + lane;
                const int64_t t = t_begin + int64_t(j) * 128 + row;
                if (j < nblk && t < t_end &&
                    SSD_IDX_OK(p.err, int64_t(b) * p.dt_sb + h + t * p.dt_sl, p.n_dt))
                    ptx::cp_async4(dst + row, dtp + t * p.dt_sl);
                else dst[row] = 0.f;
            }
            ptx::cp_async_commit();   // one group per record, empty past the end
        };
        for (int j = 0; j < 4; ++j) fetch_dt(j);
        // the states-only pass needs no C
        int kb = 0, kc = states_only ? nblk : 0, kx = 0, kr = 0;   // next block of each stream
        const int kx_end = states_only ? nblk : (nblk < 3 ? nblk : 3);
        uint64_t idle_since = 0;
        while (kb < nblk || kc < nblk || kx < kx_end || kr < nblk) {
            int fired = 0;   // bit i: stream i issued (lane 0's decision)
            if (lane == 0) {
                // B: read by C B^T(k - 2) and B^T (w o x)(k - 2)
                if (kb < nblk) {
                    const int s = kb & 1;
                    const uint32_t pp = ((kb >> 1) - 1) & 1;
                    if (kb < 2 || ((states_only || ptx::mbar_test_wait(&cb_done[s], pp)) &&
                                   ptx::mbar_test_wait(&s_done[s], pp))) {
                        const int t0 = int(t_begin + int64_t(kb) * 128);
                        ptx::mbar_arrive_expect_tx(&full_B[s], 32768);
                        ptx::tma_load_4d(smem + SM::kB + s * 32768, &tm_b, &full_B[s], 0, g, t0, b);
                        ptx::tma_load_4d(smem + SM::kB + s * 32768 + 16384, &tm_b, &full_B[s], 64,
                                         g, t0, b);
                        fired |= 1;
                    }
                }
                // C: read by C B^T(k - 2) and C h^T(k - 2), issued after it
                if (kc < nblk) {
                    const int s = kc & 1;
                    const uint32_t pp = ((kc >> 1) - 1) & 1;
                    if (kc < 2 || ptx::mbar_test_wait(&inter_done[s], pp)) {
                        const int t0 = int(t_begin + int64_t(kc) * 128);
                        ptx::mbar_arrive_expect_tx(&full_C[s], 32768);
                        ptx::tma_load_4d(smem + SM::kC + s * 32768, &tm_c, &full_C[s], 0, g, t0, b);
                        ptx::tma_load_4d(smem + SM::kC + s * 32768 + 16384, &tm_c, &full_C[s], 64,
                                         g, t0, b);
                        fired |= 2;
                    }
                }
                // x: its slot holds y(k - 3) until that tile's store has read it;
                // past the first three blocks the storer of y(k - 3) issues x(k)
                // itself (the states-only pass has no y)
                if (kx < (states_only ? nblk : (nblk < 3 ? nblk : 3))) {
                    const int slot = kx % 3;
                    if (kx < 3 || ptx::mbar_test_wait(&xfree[slot], ((kx / 3) - 1) & 1)) {
                        const int t0 = int(t_begin + int64_t(kx) * 128);
                        ptx::mbar_arrive_expect_tx(&full_X[slot], 16384);
                        ptx::tma_load_4d(smem + SM::kX + slot * 16384, &tm_x, &full_X[slot], 0, h,
                                         t0, b);
                        fired |= 4;
                    }
                }
                // the record of block k - 4 is in use until every reader released it
                if (kr < nblk &&
                    (kr < kNRec || ptx::mbar_test_wait(&rec_free[kr & 3], ((kr >> 2) - 1) & 1)))
                    fired |= 8;
                if (fired) {
                    idle_since = 0;
                } else {
                    const uint64_t now = ptx::globaltimer_ns();
                    if (!idle_since) idle_since = now;
                    else if (now - idle_since > 2000000000ull) fired = -1;
                }
            }
            fired = __shfl_sync(0xffffffffu, fired, 0);
            if (fired < 0) { ok = false; break; }
            kb += fired & 1;
            kc += (fired >> 1) & 1;
            kx += (fired >> 2) & 1;
            if (fired & 8) {
                ptx::cp_async_wait<3>();   // the group of record kr has landed
                float dtv[4];
#pragma unroll
                for (int qq = 0; qq < 4; ++qq) dtv[qq] = dtring[128 * (kr & 3) + 32 * qq + lane];
                fetch_dt(kr + 4);
                build_record(dtv, Ah, lane, rec_all + kRec * (kr & 3));
                ptx::mbar_arrive(&sc_ready[kr & 3]);
                ++kr;
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer (event loop) ----------------
        if (lane == 0 && nblk > 0) {
            // Descriptor bases, computed once: an operand at byte offset o from its
            // base is the base descriptor plus o >> 4 (start-address field; shared
            // addresses stay below 2^18, so no carry leaves the field).
            const uint64_t dCk = ptx::sdesc(ptx::smem_u32(smem + SM::kC), 16, 1024);
            const uint64_t dBk = ptx::sdesc(ptx::smem_u32(smem + SM::kB), 16, 1024);
            const uint64_t dBmn = ptx::sdesc(ptx::smem_u32(smem + SM::kB), 16384, 1024);
            const uint64_t dX = ptx::sdesc(ptx::smem_u32(smem + SM::kX), 16384, 1024);
            const uint64_t dXP = ptx::sdesc(ptx::smem_u32(smem + SM::kXP), 16384, 1024);
            const uint64_t dHB = ptx::sdesc(ptx::smem_u32(smem + SM::kHB), 16384, 1024);
            // K-major C / B over the state: K step 16 = 32 bytes, second 64-block 16 KB on
            constexpr uint32_t kKoff[8] = {0, 2, 4, 6, 1024, 1026, 1028, 1030};
            // the states-only pass issues B^T (w o x) alone
            const int k0 = states_only ? nblk : 0;
            int k_s = 0, k_in = k0, k_a = k0, k_cb = k0;   // next block of each product
            uint64_t idle_since = 0;
            // Each pass checks the products in the order L x, B^T (w o x), C h^T,
            // C B^T and issues every one that is ready (an issue takes about as
            // long as the product runs); measured the fastest of the orders tried.
            while (states_only ? k_s < nblk : (k_in < nblk || k_a < nblk)) {
                bool progress = false;
                // L x(k): the decay operand is built (after S^T(k) in issue order, so
                // that intra_done also covers S^T)
                if (k_a < k_cb && k_a < k_s) {
                    const int s = k_a & 1;
                    const uint32_t par = (k_a >> 1) & 1;
                    if (ptx::mbar_test_wait(&L_ready[s], par)) {
                        ptx::tc_fence_after();
                        const uint64_t x0 = dX + uint64_t((k_a % 3) * 1024);
                        const uint32_t t_l = tmem + 128 * s;
#pragma unroll
                        for (int ks = 0; ks < 8; ++ks)
                            ptx::mma_bf16_ts(t_l + 64, t_l + ks * 8, x0 + uint64_t(ks * 128), kIdKmn,
                                             ks != 0);
                        ptx::mma_commit(&intra_done[s]);
                        ++k_a;
                        progress = true;
                    }
                }
                // S^T(k) = B^T (w o x): w o x written, B landed, and S^T(k - 2)
                // absorbed into the state
                if (k_s < nblk) {
                    const int s = k_s & 1;
                    const uint32_t par = (k_s >> 1) & 1;
                    if (ptx::mbar_test_wait(xp_ready, k_s & 1) && ptx::mbar_test_wait(&full_B[s], par) &&
                        (k_s < 2 || ptx::mbar_test_wait(&st_done[s], par ^ 1))) {
                        ptx::tc_fence_after();
                        const uint64_t bmn0 = dBmn + uint64_t(s * 2048);
#pragma unroll
                        for (int ks = 0; ks < 8; ++ks)   // MN-major operands: K step 16 rows = 2 KB
                            ptx::mma_bf16_ss(tmem + 256 + 64 * s, bmn0 + uint64_t(ks * 128),
                                             dXP + uint64_t(ks * 128), kIdMnmn, ks != 0);
                        ptx::mma_commit(&s_done[s]);
                        ++k_s;
                        progress = true;
                    }
                }
                // C h^T(k): the state entering block k is in its operand buffer and
                // the inter accumulator of block k - 2 has been drained
                if (k_in < k_cb) {
                    const int s = k_in & 1;
                    const uint32_t par = (k_in >> 1) & 1;
                    if ((k_in == 0 || ptx::mbar_test_wait(&st_done[s ^ 1], ((k_in - 1) >> 1) & 1)) &&
                        (k_in < 2 || ptx::mbar_test_wait(&drain_done[s], par ^ 1))) {
                        ptx::tc_fence_after();
                        const uint64_t c0 = dCk + uint64_t(s * 2048);
#pragma unroll
                        for (int ks = 0; ks < 8; ++ks)
                            ptx::mma_bf16_ss(tmem + 384 + 64 * s, c0 + kKoff[ks],
                                             dHB + uint64_t(ks * 128), kIdKmn, ks != 0);
                        ptx::mma_commit(&inter_done[s]);
                        ++k_in;
                        progress = true;
                    }
                }
                // C B^T(k): its operands landed and its stage's tensor memory is free
                // (block k - 2 drained, which waited for L x(k - 2))
                if (k_cb < nblk) {
                    const int s = k_cb & 1;
                    const uint32_t par = (k_cb >> 1) & 1;
                    if (ptx::mbar_test_wait(&full_C[s], par) && ptx::mbar_test_wait(&full_B[s], par) &&
                        (k_cb < 2 || ptx::mbar_test_wait(&drain_done[s], par ^ 1))) {
                        ptx::tc_fence_after();
                        const uint64_t c0 = dCk + uint64_t(s * 2048), b0 = dBk + uint64_t(s * 2048);
#pragma unroll
                        for (int ks = 0; ks < 8; ++ks)
                            ptx::mma_bf16_ss(tmem + 128 * s, c0 + kKoff[ks], b0 + kKoff[ks], kIdCB,
                                             ks != 0);
                        ptx::mma_commit(&cb_done[s]);
                        ++k_cb;
                        progress = true;
                    }
                }
                if (progress) {
                    idle_since = 0;
                } else {
                    const uint64_t now = ptx::globaltimer_ns();
                    if (!idle_since) idle_since = now;
                    else if (now - idle_since > 2000000000ull) { ok = false; break; }
                }
            }
            // every product must land before tensor memory is released
            const int kl = nblk - 1;
            if constexpr (states_only) {
                if (ok && !ptx::mbar_wait(&s_done[kl & 1], (kl >> 1) & 1)) ok = false;
            } else {
                if (ok && !ptx::mbar_wait(&intra_done[kl & 1], (kl >> 1) & 1)) ok = false;
                if (ok && !ptx::mbar_wait(&inter_done[kl & 1], (kl >> 1) & 1)) ok = false;
            }
        }
    } else if (warp < 8) {
        // ---------------- warpgroup A: the decay operand ----------------
        // Warps 2..5 cover lane quarters 2, 3, 0, 1; warps 6, 7 add a second warp
        // to quarters 2 and 3, whose rows have the most nonzero column blocks.  A
        // warp of quarter 0 or 1 owns all four column blocks of its rows, a warp of
        // quarter 2 or 3 owns blocks {half, half + 2}: at most two nonzero blocks
        // per warp.  L block c (16 columns of bf16 pairs) overwrites the first or
        // second half of C B^T block c / 2, and blocks past the diagonal block q
        // are zero.  In a shared quarter the only cross-warp overwrites are L block
        // 1 over C B^T block 0 and L block 2 over C B^T block 1, the first block
        // each warp reads: both warps read that block, meet, then go block by block.
        const int q = warp & 3;
        const int half = (warp - 2) >> 2;          // 0 for warps 2..5, 1 for 6, 7
        const bool pair = q >= 2;
        const int cfirst = pair ? half : 0, cstep = pair ? 2 : 1, nb = pair ? 2 : 4;
        const int r = 32 * q + lane;
        const uint32_t lane_off = uint32_t(32 * q) << 16;
        const float Dh = p.D && SSD_IDX_OK(p.err, h, p.H) ? p.D[h] : 0.f;
        for (int k = 0; k < (states_only ? 0 : nblk); ++k) {
            const int s = k & 1;
            const uint32_t par = (k >> 1) & 1;
            if (!__all_sync(0xffffffffu, ptx::mbar_wait(&sc_ready[k & 3], (k >> 2) & 1) &&
                                             ptx::mbar_wait(&cb_done[s], par))) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            const float *rec = rec_all + kRec * (k & 3);
            const float gr = rec[r];
            const uint32_t tL = tmem + 128 * s + lane_off;
            uint32_t v[32], out[16];
            if (pair) {
                ptx::tmem_ld32(tL + 32 * half, v);
                ptx::tmem_ld_wait();
                ptx::tc_fence_before();
                asm volatile("bar.sync %0, 64;" ::"r"(4 + q) : "memory");
                ptx::tc_fence_after();
            }
#pragma unroll 1
            for (int i = 0; i < nb; ++i) {
                const int c = cfirst + i * cstep;
                if (c <= q) {
                    if (!pair || i > 0) {
                        ptx::tmem_ld32(tL + 32 * c, v);
                        ptx::tmem_ld_wait();
                    }
                    l_block(v, 32 * c, c == q, r, gr, ex2(gr - rec[384 + (c & 3)]), rec + 128,
                            rec + 256, Dh, out);
                } else {
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) out[jj] = 0u;
                }
                ptx::tmem_st16(tL + 16 * c, out);
            }
            ptx::tmem_st_wait();
            ptx::tc_fence_before();
            ptx::mbar_arrive(&L_ready[s]);
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&rec_free[k & 3]);
        }
    } else if (warp < 12) {
        // ---------------- warpgroup S: w o x and the carried state ----------------
        const int q = warp & 3;
        const int r = 32 * q + lane;
        const uint32_t lane_off = uint32_t(32 * q) << 16;
        uint8_t *hb = smem + SM::kHB;
        uint8_t *xprow = smem + SM::kXP + r * 128;
        // g_end of the record consumed last, kept for that block's state update
        float gend_k = 0.f;
        // w o x(k), row r, into the single w o x buffer
        auto build_wx = [&](int k) -> bool {
            if (!__all_sync(0xffffffffu, ptx::mbar_wait(&sc_ready[k & 3], (k >> 2) & 1) &&
                                             ptx::mbar_wait(&full_X[k % 3], (k / 3) & 1)))
                return false;
            const float *rec = rec_all + kRec * (k & 3);
            gend_k = rec[388];
            const float w = ex2(gend_k + rec[128 + r]);   // 2^(g_end - g_r) dt_r
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&rec_free[k & 3]);
            const __nv_bfloat162 wb = __floats2bfloat162_rn(w, w);
            const uint8_t *xrow = smem + SM::kX + (k % 3) * 16384 + r * 128;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const int off = (c ^ (r & 7)) << 4;   // swizzled: conflict-free per 8 rows
                uint4 v = *reinterpret_cast<const uint4 *>(xrow + off);
                __nv_bfloat162 *v2 = reinterpret_cast<__nv_bfloat162 *>(&v);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) v2[kk] = __hmul2(v2[kk], wb);
                *reinterpret_cast<uint4 *>(xprow + off) = v;
            }
            ptx::fence_proxy_async_smem();
            ptx::mbar_arrive(xp_ready);
            if constexpr (states_only) {   // x(k) has no other reader: release its slot
                asm volatile("bar.sync 11, 128;" ::: "memory");
                if (warp == 8 && lane == 0) ptx::mbar_arrive(&xfree[k % 3]);
            }
            return true;
        };
        if (nblk > 0 && !build_wx(0)) ok = false;
        float gend_cur = gend_k;
        [[maybe_unused]] float gsum = 0.f;   // log2 decay of the whole unit (states-only pass)
        for (int k = 0; k < nblk && ok; ++k) {
            const int s = k & 1;
            const uint32_t par = (k >> 1) & 1;
            // B^T (w o x)(k) has completed: first w o x(k + 1), which lets the next
            // S^T go to the tensor cores, then the state update
            if (!__all_sync(0xffffffffu, ptx::mbar_wait(&s_done[s], par))) {
                ok = false;
                break;
            }
            if (k + 1 < nblk && !build_wx(k + 1)) {
                ok = false;
                break;
            }
            const float gend = gend_cur;
            gend_cur = gend_k;
            if constexpr (states_only) gsum += gend;
            // h(k + 1) = 2^(g_end) h(k) + S(k); its bf16 copy replaces the one
            // C h^T(k) read
            if constexpr (!states_only) {
                if (!__all_sync(0xffffffffu, ptx::mbar_wait(&inter_done[s], par))) {
                    ok = false;
                    break;
                }
            }
            ptx::tc_fence_after();
            const float dend = ex2(gend);
            const float2 d2 = make_float2(dend, dend);
#pragma unroll
            for (int cb = 0; cb < 2; ++cb) {
                uint32_t sv[32];
                ptx::tmem_ld32(tmem + 256 + 64 * s + lane_off + 32 * cb, sv);
                ptx::tmem_ld_wait();
#pragma unroll
                for (int m = 0; m < 16; ++m)
                    hreg[16 * cb + m] = __ffma2_rn(
                        d2, hreg[16 * cb + m],
                        make_float2(__uint_as_float(sv[2 * m]), __uint_as_float(sv[2 * m + 1])));
            }
            if constexpr (!states_only) {
                if (k + 1 < nblk) write_state_row(hb, r, hreg);
            }
            ptx::fence_proxy_async_smem();
            ptx::tc_fence_before();
            ptx::mbar_arrive(&st_done[s]);
        }
        float *hout;
        if constexpr (kMode == 0)
            hout = p.h_final ? p.h_final + slab * 8192 : nullptr;
        else
            hout = unit_h_out<kMode>(p, sp, slab);
        if (hout && !((kMode == 2 && SSD_SPAN_OK(p.err, hout, sp.seg_state, sp.n_seg_state, 8192)) ||
                      (kMode != 2 && SSD_SPAN_OK(p.err, hout, p.h_final, p.n_hs, 8192))))
            hout = nullptr;
        if (ok && hout) {
#pragma unroll
            for (int m = 0; m < 32; ++m) {
                hout[(2 * m) * 128 + r] = hreg[m].x;
                hout[(2 * m + 1) * 128 + r] = hreg[m].y;
            }
        }
        if constexpr (states_only) {
            if (ok && warp == 8 && lane == 0 && SSD_IDX_OK(p.err, blockIdx.x, sp.n_seg_decay))
                sp.seg_decay[blockIdx.x] = gsum;
        }
    } else {
        // ---------------- warpgroup Y: y and its TMA store ----------------
        const int q = warp & 3;
        const int r = 32 * q + lane;
        const uint32_t lane_off = uint32_t(32 * q) << 16;
        const bool storer = (warp == 12 && lane == 0);
        for (int k = 0; k < (states_only ? 0 : nblk); ++k) {
            const int s = k & 1;
            const uint32_t par = (k >> 1) & 1;
            // y(k) = 2^(g_i) inter + intra, staged over x(k) (read by w o x and L x
            // by now) and stored as one tile by TMA (rows past the sequence end are
            // clipped)
            if (!__all_sync(0xffffffffu, ptx::mbar_wait(&sc_ready[k & 3], (k >> 2) & 1) &&
                                             ptx::mbar_wait(&inter_done[s], par) &&
                                             ptx::mbar_wait(&intra_done[s], par))) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            const float e_i = ex2(rec_all[kRec * (k & 3) + r]);
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&rec_free[k & 3]);
            const float2 e2 = make_float2(e_i, e_i);
            uint8_t *tile = smem + SM::kX + (k % 3) * 16384;
            uint8_t *row = tile + r * 128;
#pragma unroll
            for (int cb = 0; cb < 2; ++cb) {
                uint32_t a[32], d[32];
                ptx::tmem_ld32(tmem + 384 + 64 * s + lane_off + 32 * cb, a);
                ptx::tmem_ld32(tmem + 128 * s + 64 + lane_off + 32 * cb, d);
                ptx::tmem_ld_wait();
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4) {
                    const int ch = 4 * cb + c4;
                    uint32_t o[4];
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const int jj = 8 * c4 + 2 * kk;
                        const float2 acc = __ffma2_rn(
                            make_float2(__uint_as_float(a[jj]), __uint_as_float(a[jj + 1])), e2,
                            make_float2(__uint_as_float(d[jj]), __uint_as_float(d[jj + 1])));
                        o[kk] = pack_bf16(acc.x, acc.y);
                    }
                    *reinterpret_cast<uint4 *>(row + ((ch ^ (r & 7)) << 4)) =
                        make_uint4(o[0], o[1], o[2], o[3]);
                }
            }
            ptx::tc_fence_before();
            ptx::mbar_arrive(&drain_done[s]);
            ptx::fence_proxy_async_smem();
            asm volatile("bar.sync 9, 128;" ::: "memory");
            if (storer) {
                ptx::tma_store_4d(&tm_y, tile, 0, h, int(t_begin + int64_t(k) * 128), b);
                ptx::bulk_commit_group();
                ptx::bulk_wait_group_read0();   // the slot takes x(k + 3) next
                if (k + 3 < nblk) {
                    ptx::mbar_arrive_expect_tx(&full_X[k % 3], 16384);
                    ptx::tma_load_4d(tile, &tm_x, &full_X[k % 3], 0, h,
                                     int(t_begin + int64_t(k + 3) * 128), b);
                }
            }
        }
        if (storer) ptx::bulk_wait_group0();
    }
    if (!ok) atomicOr(s_err, 1);
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, kCols);
    }
    if (threadIdx.x == 0 && *s_err) atomicOr(p.err, kErrTimeout);
}

}  // namespace

bool fused_supported(const Dims &d, int xdt) {
    return xdt == DT_BF16 && d.P == 64 && d.N == 128 && d.Q % 128 == 0;
}

int device_sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
        cudaGetLastError();
        return 152;   // a GB300 (describing a plan without a device)
    }
    return n;
}

// With at least one slab per SM the run takes about (total blocks / SMs)
// block-times whatever the order (a CTA's blocks slow down as more SMs run),
// so splitting would only add work.  With fewer slabs than SMs, most SMs
// would sit idle: each slab is then split by sequence into nseg segments, at
// the price of a states-only pass over the first nseg - 1 segments (its state
// chain takes about a full block's time per block) plus a combine and two
// more launches (about 16 blocks), when that shortens the run.  Costs are in
// units of one 128-token block of the fused kernel.  Splits whose workspace
// would pass kSplitWsMax are not considered.  The general form keeps
// n_whole whole slabs ahead of the split ones.  SSD_NO_SPLIT=1 turns it off
// (comparisons).
FusedSplit fused_split(const Dims &d, int sm_count) {
    static const bool no_split = [] {
        const char *e = std::getenv("SSD_NO_SPLIT");
        return e && e[0] == '1';
    }();
    FusedSplit f{};
    const int64_t S = d.B * d.H;
    const int64_t nblk = (d.L + 127) / 128;
    const int64_t M = sm_count > 0 ? sm_count : 152;
    f.n_whole = S;
    f.tail = 0;
    f.nseg = 1;
    f.seg_len = nblk * 128;
    const int64_t full = 0, tail = S;
    if (no_split || S >= M || nblk < 2) return f;
    double best = double((S + M - 1) / M) * double(nblk);
    for (int64_t ns = 2; ns <= 64 && ns <= nblk; ++ns) {
        const int64_t bps = (nblk + ns - 1) / ns;          // blocks per segment
        const int64_t nseg = (nblk + bps - 1) / bps;        // no empty segment
        if (nseg < 2) continue;
        if (size_t(tail) * size_t(2 * nseg - 1) * size_t(d.P) * d.N * 4 + size_t(tail) * nseg * 4 +
                3 * 256 > kSplitWsMax)
            continue;
        const double cost = double(full / M) * double(nblk) +
                            double((tail * nseg + M - 1) / M) * double(bps) +
                            double((tail * (nseg - 1) + M - 1) / M) * double(bps) + 16.0;
        if (cost < best) {
            best = cost;
            f.n_whole = full;
            f.tail = tail;
            f.nseg = int(nseg);
            f.seg_len = bps * 128;
        }
    }
    if (f.nseg > 1) {
        const size_t PN = size_t(d.P) * d.N;
        auto a256 = [](size_t v) { return (v + 255) & ~size_t(255); };
        f.off_state = 0;
        f.off_decay = a256(f.off_state + size_t(f.tail) * (f.nseg - 1) * PN * 4);
        f.off_hin = a256(f.off_decay + size_t(f.tail) * (f.nseg - 1) * 4);
        f.ws_bytes = a256(f.off_hin + size_t(f.tail) * f.nseg * PN * 4);
    }
    return f;
}

namespace {
// Entering state of every tail segment s >= 1, from the states-only pass:
// h_in[s + 1] = 2^(decay_s) h_in[s] + local_s, with h_in[0] the slab's initial
// state -- the associative combine of (decay, state) pairs of "mamba-metal",
// "The essence of selective scan", in sequence order.  grid (tail, P N / 256).
__global__ void __launch_bounds__(256)
k_seg_combine(const float *h0, const float *seg_state, const float *seg_decay, float *seg_hin,
              int n_whole, int nseg, unsigned int *err, int64_t n_hs, int64_t n_state,
              int64_t n_decay, int64_t n_hin) {
    constexpr size_t PN = 8192;
    const int ts = blockIdx.x;
    const size_t e = size_t(blockIdx.y) * 256 + threadIdx.x;
    const size_t slab = size_t(n_whole) + ts;
    float hv = h0 && SSD_IDX_OK(err, slab * PN + e, n_hs) ? h0[slab * PN + e] : 0.f;
    // the loads of eight segments are issued together, then the chain runs
    for (int sg0 = 0; sg0 + 1 < nseg; sg0 += 8) {
        float dec[8], st[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int sg = sg0 + u;
            if (sg + 1 < nseg) {
                const size_t j = size_t(ts) * (nseg - 1) + sg;
                const bool in = SSD_IDX_OK(err, j, n_decay) && SSD_IDX_OK(err, j * PN + e, n_state);
                dec[u] = in ? seg_decay[j] : 0.f;
                st[u] = in ? seg_state[j * PN + e] : 0.f;
            }
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int sg = sg0 + u;
            if (sg + 1 < nseg) {
                hv = fmaf(exp2f(dec[u]), hv, st[u]);
                const size_t o = (size_t(ts) * nseg + sg + 1) * PN + e;
                if (SSD_IDX_OK(err, o, n_hin)) seg_hin[o] = hv;
            }
        }
    }
}
}  // namespace

cudaError_t launch_fused(const Args &a, cudaStream_t s) {
    const Dims &d = a.d;
    CUtensorMap tm_x, tm_b, tm_c, tm_y;
    const uint32_t box[4] = {64, 1, 128, 1};
    const uint64_t xd[4] = {64, uint64_t(d.H), uint64_t(d.L), uint64_t(d.B)};
    const uint64_t xs[3] = {uint64_t(a.x_sh) * 2, uint64_t(a.x_sl) * 2, uint64_t(a.x_sb) * 2};
    const uint64_t bd[4] = {128, uint64_t(d.G), uint64_t(d.L), uint64_t(d.B)};
    const uint64_t bs[3] = {uint64_t(a.b_sg) * 2, uint64_t(a.b_sl) * 2, uint64_t(a.b_sb) * 2};
    const uint64_t cs[3] = {uint64_t(a.c_sg) * 2, uint64_t(a.c_sl) * 2, uint64_t(a.c_sb) * 2};
    const uint64_t ys[3] = {uint64_t(a.y_sh) * 2, uint64_t(a.y_sl) * 2, uint64_t(a.y_sb) * 2};
    cudaError_t e = make_tmap_bf16(&tm_x, a.x, 4, xd, xs, box);
    if (e != cudaSuccess) return e;
    if ((e = make_tmap_bf16(&tm_b, a.Bm, 4, bd, bs, box)) != cudaSuccess) return e;
    if ((e = make_tmap_bf16(&tm_c, a.Cm, 4, bd, cs, box)) != cudaSuccess) return e;
    if ((e = make_tmap_bf16(&tm_y, a.y, 4, xd, ys, box)) != cudaSuccess) return e;
    unsigned int *err = nullptr;
    if ((e = device_error_word(&err)) != cudaSuccess) return e;
    const FusedSplit f = fused_split(d, device_sm_count());
    FusedParams p{};
    SplitParams sp{};
    p.L = d.L;
    p.seg_len = f.seg_len;
    p.B = int(d.B);
    p.H = int(d.H);
    p.hpg = int(d.hpg());
    sp.n_whole = int(f.n_whole);
    p.nseg = f.nseg;
    p.dt = a.dt;
    p.dt_sb = a.dt_sb;
    p.dt_sl = a.dt_sl;
    p.A = a.A;
    p.D = a.D;
    p.h0 = a.h0;
    p.h_final = a.final_states;
    if (f.nseg > 1) {
        sp.seg_state = reinterpret_cast<float *>(a.ws + f.off_state);
        sp.seg_decay = reinterpret_cast<float *>(a.ws + f.off_decay);
        sp.seg_hin = reinterpret_cast<const float *>(a.ws + f.off_hin);
    }
    p.y = static_cast<__nv_bfloat16 *>(a.y);
    p.y_sb = a.y_sb;
    p.y_sl = a.y_sl;
    p.y_sh = a.y_sh;
    p.err = err;
    {
        Args ax = a;
        fill_extents(ax);
        p.n_dt = ax.n_dt;
    }
    p.n_hs = d.B * d.H * 8192;
    if (f.nseg > 1) {
        sp.n_seg_state = f.tail * (f.nseg - 1) * 8192;
        sp.n_seg_decay = f.tail * (f.nseg - 1);
        sp.n_seg_hin = f.tail * f.nseg * 8192;
    }
    const int smem = FusedSmem::kBytes;
    const bool split = f.nseg > 1;
    e = split ? cudaFuncSetAttribute(k_ssd_fused<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)
              : cudaFuncSetAttribute(k_ssd_fused<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    if (f.nseg > 1) {
        // the tail segments' entering states: local states, then the combine
        e = cudaFuncSetAttribute(k_ssd_fused<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        const unsigned pre = unsigned(f.tail) * unsigned(f.nseg - 1);
        k_ssd_fused<2><<<pre, kThreads, smem, s>>>(tm_x, tm_b, tm_c, tm_y, p, sp);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        k_seg_combine<<<dim3(unsigned(f.tail), unsigned(d.P * d.N / 256)), 256, 0, s>>>(
            a.h0, sp.seg_state, sp.seg_decay, reinterpret_cast<float *>(a.ws + f.off_hin),
            sp.n_whole, f.nseg, err, p.n_hs, sp.n_seg_state, sp.n_seg_decay, sp.n_seg_hin);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    const unsigned units = unsigned(f.n_whole) + unsigned(f.tail) * unsigned(f.nseg);
    if (split)
        k_ssd_fused<1><<<units, kThreads, smem, s>>>(tm_x, tm_b, tm_c, tm_y, p, sp);
    else
        k_ssd_fused<0><<<units, kThreads, smem, s>>>(tm_x, tm_b, tm_c, tm_y, p, sp);
    return cudaGetLastError();
}

}  // namespace ssd
