// Fused SSD forward over pairs of heads: the four steps of "Accelerating
// Mamba-2 with High-Performance Forward Pass Kernels in NVIDIA CUDA Tile"
// (in-chunk cumulative sum, chunk state and its sequential pass,
// compute_out) in one kernel, one CTA per (batch, head pair) slab, for two
// heads of one group.  The chunk's C B^T is formed once per group ("Kernel 3:
// compute_out" computes cb = C B^T per group), so a CTA that owns two heads of
// a group forms it once for both, and the two heads' state and output
// products share their A operand:
//     CB    = C B^T                         N = 128, once for both heads
//     S^T   = B^T [w0 o x0 | w1 o x1]       N = 128, accumulated onto the
//                                           decayed state in tensor memory
//     inter = C [h0 | h1]^T                 N = 128
//     y_h   = 2^(g_h) o inter_h + L_h x_h   L_h x_h accumulated onto the
//                                           scaled inter in tensor memory
// A chunk of Q = 128 k tokens is evaluated as k blocks of 128 tokens joined
// through the state, as in the single-head fused kernel (ssd_fused.cu), with
// the same per-block record, decay operand and skip term on the diagonal.
//
// Tensor memory (512 columns): [128 s, +128) C B^T of the blocks of stage s
// (blocks alternate), then L_0 and L_1 written in place (32-column block c
// holds L_0 of tokens 32c.. in its first 16 columns and L_1 in its last 16),
// so that C B^T(k + 1) and its decay operand are formed while L x(k) waits for
// its inputs; [256, 384) the fp32 state of both heads (lanes = state index n,
// columns = (head, headdim)), which holds 2^(g_end) h(k) before S^T(k) adds
// onto it, so it holds h(k + 1) after; [384, 512) the y accumulator.  The
// state never leaves tensor memory: the state update is a read, one multiply
// and a write back.
//
// Roles (20 warps): warp 0 = TMA producer (B, C, x loads, y stores); warp 1 =
// tensor-memory owner and MMA issuer (one thread, an event loop); warps 2, 3 =
// the cumulative-sum record and w o x of head 0, 1; warps 4..11 = the decay
// operand (warp 4 + 4 hh + q builds L_hh on lane quarter q); warps 12..19 =
// head warps (warp 12 + 4 hh + q: the scale of inter, the state update and the
// y drain of head hh on lane quarter q).  A warp reaches tensor-memory lanes
// 32 (warp % 4) ..; every role that touches tensor memory is placed
// accordingly.
#include "ptx_sm100.cuh"
#include "ssd_block_math.cuh"
#define SSD_DBG_FILE 2u   // kDbgPair
#include "ssd_debug.cuh"
#include "ssd_internal.h"
#include "ssd_tc.cuh"
#include "ssd_tmap.h"

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdlib>

namespace ssd {
namespace {

struct PairParams {
    int64_t L;            // sequence length
    int64_t seg_len;      // tokens per tail segment (multiple of 128)
    int B, H, hpg, nseg;
    const float *dt;
    int64_t dt_sb, dt_sl;
    const float *A;
    const float *D;       // may be null
    const float *h0;      // [B][H][P][N] initial state, or null (= 0)
    float *h_final;       // [B][H][P][N] final state, or null
    unsigned int *err;
    // split launches only (see pair_split)
    const float *seg_hin; // [tail pairs][nseg][2][P][N] entering state of tail segments
    float *seg_state;     // [tail pairs][nseg - 1][2][P][N] (states-only pass)
    float *seg_decay;     // [tail pairs][nseg - 1][2]        (states-only pass)
    int n_whole;          // whole pair slabs ahead of the split ones
    // element extents, for the debug build's bounds checks
    int64_t n_dt, n_hs, n_seg_state, n_seg_decay, n_seg_hin;
};

constexpr int kPThreads = 640;   // 20 warps; 96 registers per thread
constexpr int kPRec = 392;       // floats of one head's block record (389 used)

// Shared memory.  Operand tiles first (1024-byte aligned for the 128-byte
// swizzle), then records, the dt ring and the barriers.
struct PairSmem {
    static constexpr int kC = 0;          // [128 tok][128 n] C, K-major (two 64-column halves)
    static constexpr int kB = 32768;      // [128 tok][128 n] B, K-major
    static constexpr int kX = 65536;      // 2 slots x 2 heads x [128 tok][64 p]  x, then y
    static constexpr int kW = 131072;     // 2 heads x [128 tok][64 p]          w o x
    static constexpr int kHB = 163840;    // 2 heads x [128 n][64 p]            bf16 state
    static constexpr int kF = 196608;     // 2 heads x 4 records x kPRec floats
    static constexpr int kDT = kF + 2 * 4 * kPRec * 4;   // 2 heads x 4 x [128] dt
    static constexpr int kBar = kDT + 2 * 4 * 128 * 4;
    static constexpr int kNBar = 36;
    static constexpr int kBytes = kBar + kNBar * 8 + 16;
};
static_assert(PairSmem::kBytes <= 232448, "shared memory above the per-CTA limit");
static_assert(PairSmem::kF % 16 == 0 && PairSmem::kDT % 16 == 0 && PairSmem::kBar % 8 == 0,
              "alignment");

// Tensor-memory columns.
constexpr uint32_t kTL = 0;     // C B^T / L_0, L_1, two stages of 128
constexpr uint32_t kTS = 256;   // state
constexpr uint32_t kTY = 384;   // y accumulator

// v[m] *= f for 32 fp32 values, as 16 packed multiplies.
__device__ __forceinline__ void scale32(uint32_t (&v)[32], float f) {
    const float2 f2 = make_float2(f, f);
#pragma unroll
    for (int m = 0; m < 32; m += 2) {
        const float2 r = __fmul2_rn(make_float2(__uint_as_float(v[m]), __uint_as_float(v[m + 1])), f2);
        v[m] = __float_as_uint(r.x);
        v[m + 1] = __float_as_uint(r.y);
    }
}

// A warp-uniform bounded wait: false if any lane's wait gave up.
__device__ __forceinline__ bool wait_all(uint64_t *bar, uint32_t parity) {
    return __all_sync(0xffffffffu, ptx::mbar_wait(bar, parity));
}

// Work units (kMode 0: every unit a whole pair slab; 1: whole pair slabs,
// then the tail pair slabs split into nseg segments; 2: the states-only pass
// over segments 0 .. nseg - 2 of every tail pair slab).  Pair slabs are
// numbered head pairs fastest, so neighbouring CTAs share B and C in L2.
template <int kMode>
__device__ __forceinline__ void pair_unit(const PairParams &p, int &pslab, int &seg,
                                          int64_t &t_begin, int64_t &t_end) {
    const int unit = blockIdx.x;
    if (kMode == 0 || (kMode == 1 && unit < p.n_whole)) {
        pslab = unit;
        seg = -1;
        t_begin = 0;
        t_end = p.L;
        return;
    }
    if (kMode == 2) {
        pslab = p.n_whole + unit / (p.nseg - 1);
        seg = unit % (p.nseg - 1);
    } else {
        pslab = p.n_whole + (unit - p.n_whole) / p.nseg;
        seg = (unit - p.n_whole) % p.nseg;
    }
    t_begin = int64_t(seg) * p.seg_len;
    t_end = t_begin + p.seg_len < p.L ? t_begin + p.seg_len : p.L;
}

// Barriers (index into the barrier array).  Commit barriers (one arrive from
// tcgen05.commit) mark a product's completion; the others count arrivals.
enum : int {
    kFullB = 0, kFullC = 1,            // TMA landed (single buffers)
    kCbDone = 2,                       // [2] C B^T(k) completed (stage k & 1)
    kSDone = 4,                        // S^T(k) completed
    kLReady = 5,                       // [2] L(k) built (256 threads)
    kWReady = 7,                       // w o x(k) written (64 threads: the record warps)
    kSReady = 8,                       // 2^(g_end) h(k) in the state columns (256 threads)
    kHbReady = 9,                      // bf16 h(k) written (256 threads)
    kInterDone = 10,                   // C h^T(k) completed
    kScaled = 11,                      // inter(k) scaled in place (256 threads)
    kIntraDone = 12,                   // [2] L x(k) completed: y(k) complete (stage k & 1)
    kYFree = 14,                       // y(k) read out of tensor memory (256 threads)
    kFullX = 15,                       // [2] x(k) landed in slot k & 1
    kSlotDone = 17,                    // [2] slot k & 1: y(k) staged in it (256 threads), or
                                       // in the states-only pass w o x(k) has read x(k) (64)
    kScReady = 19,                     // [2 heads][4] record ready (32 lanes)
    kRecFree = 27,                     // [2 heads][4] record released by its readers
};

template <int kMode>
__global__ void __launch_bounds__(kPThreads, 1)
k_ssd_pair(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_b,
           const __grid_constant__ CUtensorMap tm_c, const __grid_constant__ CUtensorMap tm_y,
           const PairParams p) {
    using SM = PairSmem;
    constexpr bool states_only = kMode == 2;
    constexpr uint32_t kIdCB = ptx::idesc_bf16_f32(128, 128, false, false);
    constexpr uint32_t kIdS = ptx::idesc_bf16_f32(128, 128, true, true);
    constexpr uint32_t kIdCH = ptx::idesc_bf16_f32(128, 128, false, true);
    constexpr uint32_t kIdLX = ptx::idesc_bf16_f32(128, 64, false, true);
    extern __shared__ __align__(1024) uint8_t smem[];
    if (ptx::smem_u32(smem) & 1023u) {   // uniform over the CTA: nothing has started yet
        if (threadIdx.x == 0) atomicOr(p.err, kErrSmemAlign);
        return;
    }
    float *rec_all = reinterpret_cast<float *>(smem + SM::kF);   // [2][4][kPRec]
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + SM::kBar);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + SM::kNBar);
    int *s_err = reinterpret_cast<int *>(tmem_slot + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    int pslab, seg;
    int64_t t_begin, t_end;
    pair_unit<kMode>(p, pslab, seg, t_begin, t_end);
    const int npairs = p.H >> 1;
    const int b = pslab / npairs;
    const int h_base = 2 * (pslab % npairs);
    const int g = h_base / p.hpg;
    const int nblk = int((t_end - t_begin + 127) / 128);
    if (!SSD_IN_BOUNDS(p.err, pslab >= 0 && pslab < p.B * npairs && seg < p.nseg && nblk > 0 &&
                                  t_end <= p.L && h_base + 1 < p.H))
        return;   // uniform over the CTA: nothing has started yet

    if (threadIdx.x == 0) {
        ptx::mbar_init(&bars[kFullB], 1);
        ptx::mbar_init(&bars[kFullC], 1);
        ptx::mbar_init(&bars[kSDone], 1);
        ptx::mbar_init(&bars[kWReady], 64);
        ptx::mbar_init(&bars[kSReady], 256);
        ptx::mbar_init(&bars[kHbReady], 256);
        ptx::mbar_init(&bars[kInterDone], 1);
        ptx::mbar_init(&bars[kScaled], 256);
        ptx::mbar_init(&bars[kYFree], 256);
        for (int s = 0; s < 2; ++s) {
            ptx::mbar_init(&bars[kCbDone + s], 1);
            ptx::mbar_init(&bars[kLReady + s], 256);
            ptx::mbar_init(&bars[kIntraDone + s], 1);
            ptx::mbar_init(&bars[kFullX + s], 1);
            ptx::mbar_init(&bars[kSlotDone + s], states_only ? 64 : 256);
        }
        for (int i = 0; i < 8; ++i) {
            ptx::mbar_init(&bars[kScReady + i], 32);
            // readers: the 4 decay-operand and 4 head warps of the record's head
            ptx::mbar_init(&bars[kRecFree + i], states_only ? 4 : 8);
        }
        *s_err = 0;
        ptx::fence_mbar_init();
        ptx::prefetch_tmap(&tm_x);
        ptx::prefetch_tmap(&tm_b);
        ptx::prefetch_tmap(&tm_c);
        ptx::prefetch_tmap(&tm_y);
    }
    if (warp == 1) {
        ptx::tmem_alloc(tmem_slot, 512);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    bool ok = true;

    if (warp == 0) {
        // ---------------- TMA producer and the y stores ----------------
        // Event loop: lane 0 tests the barriers and issues each stream's next
        // copy as soon as its buffer is free; the warp stays converged.  Slot
        // k & 1 holds x(k), then y(k): once y(k) is staged the producer stores
        // it, waits until the store has read the slot and loads x(k + 2) into
        // it (the states-only pass has no y: the slot is reloaded once w o x(k)
        // has read x(k)).
        auto load_x = [&](int k) {
            const int slot = k & 1;
            const int t0 = int(t_begin + int64_t(k) * 128);
            uint8_t *dst = smem + SM::kX + slot * 32768;
            ptx::mbar_arrive_expect_tx(&bars[kFullX + slot], 32768);
            ptx::tma_load_4d(dst, &tm_x, &bars[kFullX + slot], 0, h_base, t0, b);
            ptx::tma_load_4d(dst + 16384, &tm_x, &bars[kFullX + slot], 0, h_base + 1, t0, b);
            // start DRAM on the tiles three blocks on, into L2
            if (k + 3 < nblk) {
                ptx::tma_prefetch_l2_4d(&tm_x, 0, h_base, t0 + 384, b);
                ptx::tma_prefetch_l2_4d(&tm_x, 0, h_base + 1, t0 + 384, b);
            }
        };
        if (lane == 0) {
            load_x(0);
            if (nblk > 1) load_x(1);
        }
        int kb = 0, kc = states_only ? nblk : 0, ky = 0;   // next block of each stream
        uint64_t idle_since = 0;
        while (kb < nblk || kc < nblk || ky < nblk) {
            int fired = 0;
            if (lane == 0) {
                // B(k): read by C B^T(k - 1) and S^T(k - 1) until they complete
                if (kb < nblk) {
                    const int km = kb - 1;
                    if (kb == 0 ||
                        ((states_only ||
                          ptx::mbar_test_wait(&bars[kCbDone + (km & 1)], (km >> 1) & 1)) &&
                         ptx::mbar_test_wait(&bars[kSDone], km & 1))) {
                        const int t0 = int(t_begin + int64_t(kb) * 128);
                        ptx::mbar_arrive_expect_tx(&bars[kFullB], 32768);
                        ptx::tma_load_4d(smem + SM::kB, &tm_b, &bars[kFullB], 0, g, t0, b);
                        ptx::tma_load_4d(smem + SM::kB + 16384, &tm_b, &bars[kFullB], 64, g, t0, b);
                        if (kb + 2 < nblk) {   // start DRAM on the tile two blocks on
                            ptx::tma_prefetch_l2_4d(&tm_b, 0, g, t0 + 256, b);
                            ptx::tma_prefetch_l2_4d(&tm_b, 64, g, t0 + 256, b);
                        }
                        fired |= 1;
                    }
                }
                // C(k): read by C B^T(k - 1) and C h^T(k - 1)
                if (kc < nblk) {
                    const int km = kc - 1;
                    if (kc == 0 || (ptx::mbar_test_wait(&bars[kCbDone + (km & 1)], (km >> 1) & 1) &&
                                    ptx::mbar_test_wait(&bars[kInterDone], km & 1))) {
                        const int t0 = int(t_begin + int64_t(kc) * 128);
                        ptx::mbar_arrive_expect_tx(&bars[kFullC], 32768);
                        ptx::tma_load_4d(smem + SM::kC, &tm_c, &bars[kFullC], 0, g, t0, b);
                        ptx::tma_load_4d(smem + SM::kC + 16384, &tm_c, &bars[kFullC], 64, g, t0, b);
                        if (kc + 2 < nblk) {
                            ptx::tma_prefetch_l2_4d(&tm_c, 0, g, t0 + 256, b);
                            ptx::tma_prefetch_l2_4d(&tm_c, 64, g, t0 + 256, b);
                        }
                        fired |= 2;
                    }
                }
                // slot ky & 1 released: store y(ky) (rows past the sequence end are
                // clipped), then x(ky + 2)
                if (ky < nblk && ptx::mbar_test_wait(&bars[kSlotDone + (ky & 1)], (ky >> 1) & 1)) {
                    if constexpr (!states_only) {
                        const uint8_t *src = smem + SM::kX + (ky & 1) * 32768;
                        const int t0 = int(t_begin + int64_t(ky) * 128);
                        ptx::tma_store_4d(&tm_y, src, 0, h_base, t0, b);
                        ptx::tma_store_4d(&tm_y, src + 16384, 0, h_base + 1, t0, b);
                        ptx::bulk_commit_group();
                        ptx::bulk_wait_group_read0();
                    }
                    if (ky + 2 < nblk) load_x(ky + 2);
                    fired |= 4;
                }
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
            ky += (fired >> 2) & 1;
        }
        if (lane == 0) ptx::bulk_wait_group0();   // every y store has completed
    }
    else if (warp == 1) {
        // ---------------- MMA issuer (event loop, one thread) ----------------
        if (lane == 0 && nblk > 0) {
            // descriptor bases; an operand at byte offset o is the base plus o >> 4
            const uint64_t dCk = ptx::sdesc(ptx::smem_u32(smem + SM::kC), 16, 1024);
            const uint64_t dBk = ptx::sdesc(ptx::smem_u32(smem + SM::kB), 16, 1024);
            const uint64_t dBmn = ptx::sdesc(ptx::smem_u32(smem + SM::kB), 16384, 1024);
            const uint64_t dW = ptx::sdesc(ptx::smem_u32(smem + SM::kW), 16384, 1024);
            const uint64_t dHB = ptx::sdesc(ptx::smem_u32(smem + SM::kHB), 16384, 1024);
            const uint64_t dX = ptx::sdesc(ptx::smem_u32(smem + SM::kX), 16384, 1024);
            // K-major C / B over the state: K step 16 = 32 bytes, second half 16 KB on
            constexpr uint32_t kKoff[8] = {0, 2, 4, 6, 1024, 1026, 1028, 1030};
            // next block of each product (the states-only pass issues S^T alone)
            int k_cb = states_only ? nblk : 0, k_ch = states_only ? nblk : 0, k_s = 0,
                k_lx = states_only ? nblk : 0;
            uint64_t idle_since = 0;
            // Every test names a phase that cannot be confused with an earlier one
            // of the same parity: the product two phases back is already issued.
            while (k_lx < nblk || k_s < nblk) {
                bool progress = false;
                // L x(k): L(k) built, inter(k) scaled, x(k) landed
                if (k_lx < k_cb && k_lx < k_ch) {
                    const int s = k_lx & 1;
                    const uint32_t ps = (k_lx >> 1) & 1;
                    if (ptx::mbar_test_wait(&bars[kLReady + s], ps) &&
                        ptx::mbar_test_wait(&bars[kScaled], k_lx & 1) &&
                        ptx::mbar_test_wait(&bars[kFullX + s], ps)) {
                        ptx::tc_fence_after();
                        const uint64_t x0 = dX + uint64_t(s * 2048);
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh)
#pragma unroll
                            for (int ks = 0; ks < 8; ++ks)
                                ptx::mma_bf16_ts(tmem + kTY + 64 * hh,
                                                 tmem + kTL + 128 * s + 32 * (ks >> 1) + 8 * (ks & 1) +
                                                     16 * hh,
                                                 x0 + uint64_t(hh * 1024 + ks * 128), kIdLX, 1);
                        ptx::mma_commit(&bars[kIntraDone + s]);
                        ++k_lx;
                        progress = true;
                    }
                }
                // C B^T(k) into stage k & 1: B, C landed and L x(k - 2) has
                // completed (it read L(k - 2) from that stage)
                if (k_cb < nblk && (k_cb < 2 || k_lx >= k_cb - 1)) {
                    const int s = k_cb & 1;
                    if (ptx::mbar_test_wait(&bars[kFullB], k_cb & 1) &&
                        ptx::mbar_test_wait(&bars[kFullC], k_cb & 1) &&
                        (k_cb < 2 ||
                         ptx::mbar_test_wait(&bars[kIntraDone + s], ((k_cb - 2) >> 1) & 1))) {
                        ptx::tc_fence_after();
#pragma unroll
                        for (int ks = 0; ks < 8; ++ks)
                            ptx::mma_bf16_ss(tmem + kTL + 128 * s, dCk + kKoff[ks], dBk + kKoff[ks],
                                             kIdCB, ks != 0);
                        ptx::mma_commit(&bars[kCbDone + s]);
                        ++k_cb;
                        progress = true;
                    }
                }
                // C h^T(k): C landed, bf16 h(k) written, y accumulator free
                // (y(k - 1) drained)
                if (k_ch < nblk) {
                    if (ptx::mbar_test_wait(&bars[kFullC], k_ch & 1) &&
                        ptx::mbar_test_wait(&bars[kHbReady], k_ch & 1) &&
                        (k_ch == 0 || ptx::mbar_test_wait(&bars[kYFree], (k_ch - 1) & 1))) {
                        ptx::tc_fence_after();
#pragma unroll
                        for (int ks = 0; ks < 8; ++ks)   // MN-major state: K step 16 rows = 2 KB
                            ptx::mma_bf16_ss(tmem + kTY, dCk + kKoff[ks], dHB + uint64_t(ks * 128),
                                             kIdCH, ks != 0);
                        ptx::mma_commit(&bars[kInterDone]);
                        ++k_ch;
                        progress = true;
                    }
                }
                // S^T(k) onto the decayed state: B landed, w o x(k) written, state decayed
                if (k_s < nblk) {
                    if (ptx::mbar_test_wait(&bars[kFullB], k_s & 1) &&
                        ptx::mbar_test_wait(&bars[kWReady], k_s & 1) &&
                        ptx::mbar_test_wait(&bars[kSReady], k_s & 1)) {
                        ptx::tc_fence_after();
#pragma unroll
                        for (int ks = 0; ks < 8; ++ks)   // MN-major operands: K step 16 rows = 2 KB
                            ptx::mma_bf16_ss(tmem + kTS, dBmn + uint64_t(ks * 128),
                                             dW + uint64_t(ks * 128), kIdS, 1);
                        ptx::mma_commit(&bars[kSDone]);
                        ++k_s;
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
            if (ok && !ptx::mbar_wait(&bars[kSDone], kl & 1)) ok = false;
            if constexpr (!states_only) {
                if (ok && !ptx::mbar_wait(&bars[kIntraDone + (kl & 1)], (kl >> 1) & 1)) ok = false;
            }
        }
    }
    else if (warp < 4) {
        // ---------------- records and w o x of head hh ----------------
        // The block's cumulative-sum record, built three blocks ahead, and
        // w o x(k) (w_r = 2^(g_end - g_r) dt_r) into the single w o x buffer
        // once S^T(k - 1) has read it.  dt of record j is copied asynchronously
        // into ring slot j & 3, four records ahead; each lane copies, and later
        // reads, its own four rows.
        const int hh = warp - 2;
        const float Ah = SSD_IDX_OK(p.err, h_base + hh, p.H) ? p.A[h_base + hh] : 0.f;
        const float *dtp = p.dt + int64_t(b) * p.dt_sb + h_base + hh;
        float *dtring = reinterpret_cast<float *>(smem + SM::kDT) + hh * 512;
        float *rec0 = rec_all + hh * 4 * kPRec;
        auto fetch_dt = [&](int j) {
            float *dst = dtring + 128 * (j & 3);
#pragma unroll
            for (int qq = 0; qq < 4; ++qq) {
                const int row = 32 * qq + lane;
                const int64_t t = t_begin + int64_t(j) * 128 + row;
                if (j < nblk && t < t_end &&
                    SSD_IDX_OK(p.err, int64_t(b) * p.dt_sb + h_base + hh + t * p.dt_sl, p.n_dt))
                    ptx::cp_async4(dst + row, dtp + t * p.dt_sl);
                else dst[row] = 0.f;
            }
            ptx::cp_async_commit();   // one group per record, empty past the end
        };
        int kr = 0;   // next record to build
        auto build_next_record = [&]() -> bool {
            if (kr >= 4 && !wait_all(&bars[kRecFree + hh * 4 + (kr & 3)], ((kr >> 2) - 1) & 1))
                return false;
            ptx::cp_async_wait<3>();   // the group of record kr has landed
            float dtv[4];
#pragma unroll
            for (int qq = 0; qq < 4; ++qq) dtv[qq] = dtring[128 * (kr & 3) + 32 * qq + lane];
            fetch_dt(kr + 4);
            build_record(dtv, Ah, lane, rec0 + kPRec * (kr & 3));
            ptx::mbar_arrive(&bars[kScReady + hh * 4 + (kr & 3)]);
            ++kr;
            return true;
        };
        [[maybe_unused]] float gsum = 0.f;   // log2 decay of the unit (states-only pass)
        for (int j = 0; j < 4; ++j) fetch_dt(j);
        for (int j = 0; j < 3 && kr < nblk && ok; ++j) ok = build_next_record();
        for (int k = 0; k < nblk && ok; ++k) {
            const int slot = k & 1;
            if (!__all_sync(0xffffffffu,
                            ptx::mbar_wait(&bars[kFullX + slot], (k >> 1) & 1) &&
                                (k == 0 || ptx::mbar_wait(&bars[kSDone], (k - 1) & 1)))) {
                ok = false;
                break;
            }
            __syncwarp();   // this warp's record k is visible to all its lanes
            const float *rec = rec0 + kPRec * (k & 3);
            const float gend = rec[388];
            if constexpr (states_only) gsum += gend;
            const uint8_t *xt = smem + SM::kX + slot * 32768 + hh * 16384;
            uint8_t *wt = smem + SM::kW + hh * 16384;
#pragma unroll 1
            for (int i = 0; i < 4; i += 2) {
                uint4 v[2][8];
                __nv_bfloat162 wb[2];
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int r = 32 * (i + u) + lane;
                    const float w = ex2(gend + rec[128 + r]);
                    wb[u] = __floats2bfloat162_rn(w, w);
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        v[u][c] = *reinterpret_cast<const uint4 *>(xt + r * 128 + ((c ^ (r & 7)) << 4));
                }
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int r = 32 * (i + u) + lane;
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        __nv_bfloat162 *v2 = reinterpret_cast<__nv_bfloat162 *>(&v[u][c]);
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) v2[kk] = __hmul2(v2[kk], wb[u]);
                        *reinterpret_cast<uint4 *>(wt + r * 128 + ((c ^ (r & 7)) << 4)) = v[u][c];
                    }
                }
            }
            ptx::fence_proxy_async_smem();
            ptx::mbar_arrive(&bars[kWReady]);
            if constexpr (states_only) ptx::mbar_arrive(&bars[kSlotDone + slot]);   // x(k) read
            if (kr < nblk) ok = build_next_record();
        }
        ptx::cp_async_wait<0>();
        if constexpr (states_only) {
            const size_t jd = (size_t(pslab - p.n_whole) * (p.nseg - 1) + seg) * 2 + hh;
            if (ok && lane == 0 && SSD_IDX_OK(p.err, jd, p.n_seg_decay)) p.seg_decay[jd] = gsum;
        }
    } else if (warp < 12) {
        // ---------------- decay operand L_hh on lane quarter q ----------------
        // Row r's 32-column block c (c <= q) of C B^T is read by both warps of
        // quarter q, which then overwrite it with L_0 (first 16 columns) and
        // L_1 (last 16): the barrier between the read and the writes keeps
        // either warp from overwriting a block the other has not read.  Blocks
        // past the diagonal block q are zero.
        const int q = warp & 3, hh = (warp - 4) >> 2;
        const int r = 32 * q + lane;
        const uint32_t lane_off = uint32_t(32 * q) << 16;
        const float Dh = p.D && SSD_IDX_OK(p.err, h_base + hh, p.H) ? p.D[h_base + hh] : 0.f;
        const float *rec0 = rec_all + hh * 4 * kPRec;
        for (int k = 0; k < (states_only ? 0 : nblk); ++k) {
            if (!__all_sync(0xffffffffu,
                            ptx::mbar_wait(&bars[kScReady + hh * 4 + (k & 3)], (k >> 2) & 1) &&
                                ptx::mbar_wait(&bars[kCbDone + (k & 1)], (k >> 1) & 1))) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            const float *rec = rec0 + kPRec * (k & 3);
            const float gr = rec[r];
            const uint32_t t_l = tmem + kTL + 128 * (k & 1) + lane_off;
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
                uint32_t out[16];
                if (c <= q) {
                    uint32_t v[32];
                    ptx::tmem_ld32(t_l + 32 * c, v);
                    ptx::tmem_ld_wait();
                    ptx::tc_fence_before();
                    asm volatile("bar.sync %0, 64;" ::"r"(1 + q) : "memory");
                    ptx::tc_fence_after();
                    l_block(v, 32 * c, c == q, r, gr, ex2(gr - rec[384 + c]), rec + 128, rec + 256,
                            Dh, out);
                } else {
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) out[jj] = 0u;
                }
                ptx::tmem_st16(t_l + 32 * c + 16 * hh, out);
            }
            ptx::tmem_st_wait();
            ptx::tc_fence_before();
            ptx::mbar_arrive(&bars[kLReady + (k & 1)]);
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&bars[kRecFree + hh * 4 + (k & 3)]);
        }
    }
    else {
        // ---------------- head warps: head hh on lane quarter q ----------------
        const int q = warp & 3, hh = (warp - 12) >> 2;
        const int h = h_base + hh;
        const int r = 32 * q + lane;
        const uint32_t lane_off = uint32_t(32 * q) << 16;
        const float *rec0 = rec_all + hh * 4 * kPRec;
        uint8_t *hbrow = smem + SM::kHB + hh * 16384 + r * 128;
        const int ts = pslab - p.n_whole;   // tail pair slab (split launches)
        const uint32_t t_state = tmem + kTS + 64 * hh + lane_off;   // this row's 64 state columns

        // bf16 copy of 32 state values (headdim 32 cb ..) into row r of the operand tile
        auto write_hb = [&](int cb, const uint32_t (&v)[32]) {
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) {
                const int c = 4 * cb + c4;
                const uint4 u = make_uint4(
                    pack_bf16(__uint_as_float(v[8 * c4]), __uint_as_float(v[8 * c4 + 1])),
                    pack_bf16(__uint_as_float(v[8 * c4 + 2]), __uint_as_float(v[8 * c4 + 3])),
                    pack_bf16(__uint_as_float(v[8 * c4 + 4]), __uint_as_float(v[8 * c4 + 5])),
                    pack_bf16(__uint_as_float(v[8 * c4 + 6]), __uint_as_float(v[8 * c4 + 7])));
                *reinterpret_cast<uint4 *>(hbrow + ((c ^ (r & 7)) << 4)) = u;
            }
        };
        // the record's readers among the head warps: the scale of inter(k) in
        // the full pass, the state update of block k - 1 in the states-only pass
        auto release_record = [&](int k) {
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&bars[kRecFree + hh * 4 + (k & 3)]);
        };

        // the entering state: 2^(g_end(0)) h into the state columns, bf16 h into
        // the operand tile
        if (!wait_all(&bars[kScReady + hh * 4], 0)) ok = false;
        if (ok) {
            const float *hin;
            if constexpr (kMode == 2) hin = nullptr;
            else if (seg > 0) {
                const size_t o = ((size_t(ts) * p.nseg + seg) * 2 + hh) * 8192;
                hin = SSD_IDX_OK(p.err, o + 8191, p.n_seg_hin) ? p.seg_hin + o : nullptr;
            } else {
                const size_t o = (size_t(b) * p.H + h) * 8192;
                hin = p.h0 && SSD_IDX_OK(p.err, o + 8191, p.n_hs) ? p.h0 + o : nullptr;
            }
            const float d0 = ex2(rec0[388]);
            if constexpr (states_only) release_record(0);
#pragma unroll
            for (int cb = 0; cb < 2; ++cb) {
                uint32_t v[32];
#pragma unroll
                for (int m = 0; m < 32; ++m)
                    v[m] = __float_as_uint(hin ? hin[(32 * cb + m) * 128 + r] : 0.f);
                if constexpr (!states_only) write_hb(cb, v);
#pragma unroll
                for (int m = 0; m < 32; ++m) v[m] = __float_as_uint(d0 * __uint_as_float(v[m]));
                ptx::tmem_st32(t_state + 32 * cb, v);
            }
            ptx::tmem_st_wait();
            ptx::fence_proxy_async_smem();
            ptx::tc_fence_before();
            ptx::mbar_arrive(&bars[kSReady]);
            ptx::mbar_arrive(&bars[kHbReady]);
        }

        for (int k = 0; k < nblk && ok; ++k) {
            const int s = k & 1;
            const uint32_t ps = (k >> 1) & 1;
            const uint32_t t_y = tmem + kTY + 64 * hh + lane_off;   // this row's y columns
            if constexpr (!states_only) {
                // 1. inter(k) = C h^T(k), scaled in place by 2^(g_r); L x(k) adds onto it
                if (!wait_all(&bars[kInterDone], k & 1)) { ok = false; break; }
                ptx::tc_fence_after();
                const float e = ex2(rec0[kPRec * (k & 3) + r]);
                release_record(k);
#pragma unroll
                for (int cb = 0; cb < 2; ++cb) {
                    uint32_t a[32];
                    ptx::tmem_ld32(t_y + 32 * cb, a);
                    ptx::tmem_ld_wait();
                    scale32(a, e);
                    ptx::tmem_st32(t_y + 32 * cb, a);
                }
                ptx::tmem_st_wait();
                ptx::tc_fence_before();
                ptx::mbar_arrive(&bars[kScaled]);
            }
            // 2. h(k + 1) is in the state columns once S^T(k) has completed: keep
            // its bf16 copy for C h^T(k + 1) (C h^T(k) has read the old one) and
            // decay it by 2^(g_end(k + 1)) for S^T(k + 1); after the last block
            // it is the unit's final state
            if (!wait_all(&bars[kSDone], k & 1)) { ok = false; break; }
            ptx::tc_fence_after();
            const bool last = k + 1 == nblk;
            float d1 = 0.f;
            float *hout = nullptr;
            if (!last) {
                const int k1 = k + 1;
                if (!wait_all(&bars[kScReady + hh * 4 + (k1 & 3)], (k1 >> 2) & 1)) {
                    ok = false;
                    break;
                }
                d1 = ex2(rec0[kPRec * (k1 & 3) + 388]);
                if constexpr (states_only) release_record(k1);
            } else if constexpr (kMode == 2) {
                const size_t o = ((size_t(ts) * (p.nseg - 1) + seg) * 2 + hh) * 8192;
                hout = SSD_IDX_OK(p.err, o + 8191, p.n_seg_state) ? p.seg_state + o : nullptr;
            } else if (seg < 0 || seg == p.nseg - 1) {
                const size_t o = (size_t(b) * p.H + h) * 8192;
                hout = p.h_final && SSD_IDX_OK(p.err, o + 8191, p.n_hs) ? p.h_final + o : nullptr;
            }
#pragma unroll
            for (int cb = 0; cb < 2; ++cb) {
                uint32_t v[32];
                ptx::tmem_ld32(t_state + 32 * cb, v);
                ptx::tmem_ld_wait();
                if (!last) {
                    if constexpr (!states_only) write_hb(cb, v);
                    scale32(v, d1);
                    ptx::tmem_st32(t_state + 32 * cb, v);
                } else if (hout) {
#pragma unroll
                    for (int m = 0; m < 32; ++m) hout[(32 * cb + m) * 128 + r] = __uint_as_float(v[m]);
                }
            }
            if (!last) {
                ptx::tmem_st_wait();
                ptx::fence_proxy_async_smem();
                ptx::tc_fence_before();
                ptx::mbar_arrive(&bars[kSReady]);
                ptx::mbar_arrive(&bars[kHbReady]);
            }
            if constexpr (!states_only) {
                // 3. y(k) = the accumulator once L x(k) has completed: bf16 into
                // this row of head hh's tile in the x(k) slot, which the producer
                // stores once all rows are in
                if (!wait_all(&bars[kIntraDone + s], ps)) { ok = false; break; }
                ptx::tc_fence_after();
                uint8_t *yrow = smem + SM::kX + s * 32768 + hh * 16384 + r * 128;
                auto put = [&](int cb, const uint32_t (&a)[32]) {
#pragma unroll
                    for (int c4 = 0; c4 < 4; ++c4) {
                        const int c = 4 * cb + c4;
                        const uint4 u = make_uint4(
                            pack_bf16(__uint_as_float(a[8 * c4]), __uint_as_float(a[8 * c4 + 1])),
                            pack_bf16(__uint_as_float(a[8 * c4 + 2]), __uint_as_float(a[8 * c4 + 3])),
                            pack_bf16(__uint_as_float(a[8 * c4 + 4]), __uint_as_float(a[8 * c4 + 5])),
                            pack_bf16(__uint_as_float(a[8 * c4 + 6]), __uint_as_float(a[8 * c4 + 7])));
                        *reinterpret_cast<uint4 *>(yrow + ((c ^ (r & 7)) << 4)) = u;
                    }
                };
#pragma unroll
                for (int cb = 0; cb < 2; ++cb) {
                    uint32_t a[32];
                    ptx::tmem_ld32(t_y + 32 * cb, a);
                    ptx::tmem_ld_wait();
                    put(cb, a);
                }
                ptx::tc_fence_before();
                ptx::mbar_arrive(&bars[kYFree]);
                ptx::fence_proxy_async_smem();
                ptx::mbar_arrive(&bars[kSlotDone + s]);
            }
        }
    }
    if (!ok) atomicOr(s_err, 1);
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, 512);
    }
    if (threadIdx.x == 0 && *s_err) atomicOr(p.err, kErrTimeout);
}

// Entering state of every tail segment s >= 1 from the states-only pass:
// h_in(s + 1) = 2^(decay_s) h_in(s) + local_s with h_in(0) the slab's initial
// state -- the associative combine of (decay, state) pairs of "mamba-metal",
// "The essence of selective scan", in sequence order.  grid (tail pairs x 2
// heads, P N / 256).
__global__ void __launch_bounds__(256)
k_pair_combine(const float *h0, const float *seg_state, const float *seg_decay, float *seg_hin,
               int n_whole, int nseg, int H, unsigned int *err, int64_t n_hs, int64_t n_state,
               int64_t n_decay, int64_t n_hin) {
    constexpr size_t PN = 8192;
    const int ts = blockIdx.x >> 1, hh = blockIdx.x & 1;
    const size_t e = size_t(blockIdx.y) * 256 + threadIdx.x;
    const int pslab = n_whole + ts;
    const int npairs = H >> 1;
    const size_t slab = size_t(pslab / npairs) * H + 2 * (pslab % npairs) + hh;
    float hv = h0 && SSD_IDX_OK(err, slab * PN + e, n_hs) ? h0[slab * PN + e] : 0.f;
    // the loads of eight segments are issued together, then the chain runs
    for (int sg0 = 0; sg0 + 1 < nseg; sg0 += 8) {
        float dec[8], st[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int sg = sg0 + u;
            if (sg + 1 < nseg) {
                const size_t j = (size_t(ts) * (nseg - 1) + sg) * 2 + hh;
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
                const size_t o = ((size_t(ts) * nseg + sg + 1) * 2 + hh) * PN + e;
                if (SSD_IDX_OK(err, o, n_hin)) seg_hin[o] = hv;
            }
        }
    }
}

}  // namespace

bool pair_supported(const Dims &d, int xdt) {
    static const bool off = [] {
        const char *e = std::getenv("SSD_NO_PAIR");
        return e && e[0] == '1';
    }();
    // Two heads per CTA halve the number of units; with fewer pair slabs than
    // SMs the single-head kernel keeps more SMs busy (and splits by sequence
    // less), and it measured faster on every such workload.
    return !off && fused_supported(d, xdt) && d.H % 2 == 0 && d.hpg() % 2 == 0 &&
           d.B * d.H / 2 >= device_sm_count();
}

// Cost model in units of one pair-block (128 tokens of two heads) on one SM.
// Whole pair slabs run in full waves of M; the pair slabs left over (fewer
// than M) are split by sequence into nseg segments of bps blocks, after a
// states-only pass over the first nseg - 1 segments (charged kPre of a full
// block per block: it runs only S^T, w o x and the state update) and the
// combine (charged kFix blocks with the two extra launches).  Splits whose
// workspace would pass kSplitWsMax are skipped.  SSD_NO_SPLIT=1 turns
// splitting off (comparisons).
FusedSplit pair_split(const Dims &d, int sm_count) {
    static const bool no_split = [] {
        const char *e = std::getenv("SSD_NO_SPLIT");
        return e && e[0] == '1';
    }();
    constexpr double kPre = 0.5, kFix = 6.0;
    FusedSplit f{};
    const int64_t S = d.B * d.H / 2;
    const int64_t nblk = (d.L + 127) / 128;
    const int64_t M = sm_count > 0 ? sm_count : 152;
    f.n_whole = S;
    f.tail = 0;
    f.nseg = 1;
    f.seg_len = nblk * 128;
    if (no_split || nblk < 2) return f;
    const int64_t full = (S / M) * M, tail = S - full;
    if (tail == 0) return f;
    const size_t PN2 = size_t(d.P) * d.N * 2;   // one pair's state, floats
    double best = double((S + M - 1) / M) * double(nblk);
    for (int64_t ns = 2; ns <= 64 && ns <= nblk; ++ns) {
        const int64_t bps = (nblk + ns - 1) / ns;          // blocks per segment
        const int64_t nseg = (nblk + bps - 1) / bps;        // no empty segment
        if (nseg < 2) continue;
        if (size_t(tail) * size_t(2 * nseg - 1) * PN2 * 4 + size_t(tail) * nseg * 8 + 3 * 256 >
            kSplitWsMax)
            continue;
        const double cost = double(full / M) * double(nblk) +
                            double((tail * nseg + M - 1) / M) * double(bps) +
                            kPre * double((tail * (nseg - 1) + M - 1) / M) * double(bps) + kFix;
        if (cost < best) {
            best = cost;
            f.n_whole = full;
            f.tail = tail;
            f.nseg = int(nseg);
            f.seg_len = bps * 128;
        }
    }
    if (f.nseg > 1) {
        auto a256 = [](size_t v) { return (v + 255) & ~size_t(255); };
        f.off_state = 0;
        f.off_decay = a256(f.off_state + size_t(f.tail) * (f.nseg - 1) * PN2 * 4);
        f.off_hin = a256(f.off_decay + size_t(f.tail) * (f.nseg - 1) * 8);
        f.ws_bytes = a256(f.off_hin + size_t(f.tail) * f.nseg * PN2 * 4);
    }
    return f;
}

cudaError_t launch_pair(const Args &a, cudaStream_t s) {
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
    const FusedSplit f = pair_split(d, device_sm_count());
    PairParams p{};
    p.L = d.L;
    p.seg_len = f.seg_len;
    p.B = int(d.B);
    p.H = int(d.H);
    p.hpg = int(d.hpg());
    p.nseg = f.nseg;
    p.n_whole = int(f.n_whole);
    p.dt = a.dt;
    p.dt_sb = a.dt_sb;
    p.dt_sl = a.dt_sl;
    p.A = a.A;
    p.D = a.D;
    p.h0 = a.h0;
    p.h_final = a.final_states;
    p.err = err;
    {
        Args ax = a;
        fill_extents(ax);
        p.n_dt = ax.n_dt;
    }
    p.n_hs = d.B * d.H * 8192;
    if (f.nseg > 1) {
        p.n_seg_state = f.tail * (f.nseg - 1) * 2 * 8192;
        p.n_seg_decay = f.tail * (f.nseg - 1) * 2;
        p.n_seg_hin = f.tail * f.nseg * 2 * 8192;
    }
    const int smem = PairSmem::kBytes;
    if (f.nseg > 1) {
        p.seg_state = reinterpret_cast<float *>(a.ws + f.off_state);
        p.seg_decay = reinterpret_cast<float *>(a.ws + f.off_decay);
        p.seg_hin = reinterpret_cast<const float *>(a.ws + f.off_hin);
        // the tail segments' entering states: local states, then the combine
        if ((e = cudaFuncSetAttribute(k_ssd_pair<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      smem)) != cudaSuccess ||
            (e = cudaFuncSetAttribute(k_ssd_pair<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      smem)) != cudaSuccess)
            return e;
        const unsigned pre = unsigned(f.tail) * unsigned(f.nseg - 1);
        k_ssd_pair<2><<<pre, kPThreads, smem, s>>>(tm_x, tm_b, tm_c, tm_y, p);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        k_pair_combine<<<dim3(unsigned(f.tail) * 2, unsigned(d.P * d.N / 256)), 256, 0, s>>>(
            a.h0, p.seg_state, p.seg_decay, reinterpret_cast<float *>(a.ws + f.off_hin),
            p.n_whole, f.nseg, p.H, err, p.n_hs, p.n_seg_state, p.n_seg_decay, p.n_seg_hin);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        const unsigned units = unsigned(f.n_whole) + unsigned(f.tail) * unsigned(f.nseg);
        k_ssd_pair<1><<<units, kPThreads, smem, s>>>(tm_x, tm_b, tm_c, tm_y, p);
    } else {
        if ((e = cudaFuncSetAttribute(k_ssd_pair<0>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      smem)) != cudaSuccess)
            return e;
        k_ssd_pair<0><<<unsigned(f.n_whole), kPThreads, smem, s>>>(tm_x, tm_b, tm_c, tm_y, p);
    }
    return cudaGetLastError();
}

}  // namespace ssd
