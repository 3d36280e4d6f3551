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
//     inter = C h^T                                  tensor cores -> TMEM
//     L_ij  = [j <= i] CB_ij 2^(g_i - g_j) dt_j      math warps, in place in TMEM (bf16)
//     intra = L x                                    tensor cores, A read from TMEM
//     S^T   = B^T (w o x),  w_j = 2^(g_end - g_j) dt_j   tensor cores -> TMEM
//     y     = 2^(g_i) inter + intra + D x            math warps (drain)
//     h     = 2^(g_end) h + S                        math warps, fp32 in registers
// dt_j is folded into the exponent, 2^(g_i - g_j + log2 dt_j) (dt_j = 0 gives
// 2^-inf = 0), and the causal selection replaces the exponent of masked
// entries by -inf before it is evaluated, so no positive exponent of the
// decay is ever computed.
//
// The blocks of one slab are software-pipelined across two stages: only the
// fp32 state update h(k + 1) = 2^(g_end) h(k) + S(k) and the product C h^T it
// feeds are serial; C B^T, L, L x and B^T (w o x) of later blocks proceed
// while earlier blocks are drained.  Roles: warp 0 = TMA producer (128-byte
// swizzle, no multicast), warp 1 = tensor-memory owner and MMA issuer, warps
// 2..9 = warpgroup A (w o x and L), warps 10..13 = warpgroup B (state update,
// y).  A thread owns tile row / state row r = its TMEM lane.  One CTA per SM
// (512 TMEM columns, ~213 KB of shared memory).
#include "ptx_sm100.cuh"
#include "ssd_internal.h"
#include "ssd_tc.cuh"
#include "ssd_tmap.h"

#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace ssd {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

struct FusedParams {
    int64_t L;            // sequence length
    int64_t seg_len;      // tokens per segment (multiple of 128)
    int B, H, hpg, nseg;
    const float *dt;
    int64_t dt_sb, dt_sl;
    const float *A;
    const float *D;       // may be null
    const float *h_in;    // [nseg][B][H][P][N] entering state per segment, or null (= 0)
    float *h_out;         // [B][H][P][N] state after the last segment, or null
    __nv_bfloat16 *y;
    int64_t y_sb, y_sl, y_sh;
    unsigned int *err;
};

// Shared memory (one CTA per SM): two stages of the C, B and x tiles and of
// w o x, the bf16 carried-state operand, and per-stage small arrays.
struct FusedSmem {
    static constexpr int kC = 0;          // 2 stages x 2 x [128 tokens][128 B]  C, K-major
    static constexpr int kB = 65536;      // 2 stages x 2 x [128 tokens][128 B]  B, K-major
    static constexpr int kX = 131072;     // 2 stages x [128 tokens][128 B]      x, MN-major
    static constexpr int kXP = 163840;    // 2 stages x [128 tokens][128 B]      w o x
    static constexpr int kHB = 196608;    // [128 n][128 B]                      bf16 state
    static constexpr int kF = 212992;     // grow, ngd, w2, vcol [2][128]; wsum, gpiv [2][4]
    static constexpr int kBar = kF + (8 * 128 + 16) * 4;
    static constexpr int kBytes = kBar + 256 + 1024;
};

constexpr int kThreads = 448;             // 14 warps
constexpr int kWgA = 256;                 // warpgroup A threads (warps 2..9)


__device__ __forceinline__ uint8_t *align1024(uint8_t *p) {
    return reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ float2 unpack_bf16(uint32_t u) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u));
}

// 2^x with the hardware approximation (relative error ~2^-22; -inf gives +0)
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Writes this thread's state row n = r (64 headdim values, bf16) into the
// [128 n][64 p] MN-major, 128-byte-swizzled operand tile.
__device__ __forceinline__ void write_state_row(uint8_t *tile, int r, const float2 (&h)[32]) {
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        const uint4 v = make_uint4(pack_bf16(h[4 * c].x, h[4 * c].y),
                                   pack_bf16(h[4 * c + 1].x, h[4 * c + 1].y),
                                   pack_bf16(h[4 * c + 2].x, h[4 * c + 2].y),
                                   pack_bf16(h[4 * c + 3].x, h[4 * c + 3].y));
        *reinterpret_cast<uint4 *>(tile + r * 128 + ((c ^ (r & 7)) << 4)) = v;
    }
}

// One 32-column block of the decay operand for row r: entries
// cb[j] * 2^(gr + ngd[j]) with ngd[j] = log2(dt_j) - g_j, and, on the
// diagonal block, -inf exponents for j > r.
__device__ __forceinline__ void l_block(const uint32_t (&v)[32], int col0, bool diag, int r,
                                        float gr, const float *ngd, uint32_t (&out)[16]) {
    const float2 g2 = make_float2(gr, gr);
#pragma unroll
    for (int jj = 0; jj < 32; jj += 4) {
        const float4 n4 = *reinterpret_cast<const float4 *>(ngd + col0 + jj);
        float2 a0 = __fadd2_rn(g2, make_float2(n4.x, n4.y));
        float2 a1 = __fadd2_rn(g2, make_float2(n4.z, n4.w));
        if (diag) {
            const int j = col0 + jj;
            if (j > r) a0.x = -INFINITY;
            if (j + 1 > r) a0.y = -INFINITY;
            if (j + 2 > r) a1.x = -INFINITY;
            if (j + 3 > r) a1.y = -INFINITY;
        }
        const float2 e0 = __fmul2_rn(make_float2(ex2(a0.x), ex2(a0.y)),
                                     make_float2(__uint_as_float(v[jj]), __uint_as_float(v[jj + 1])));
        const float2 e1 = __fmul2_rn(make_float2(ex2(a1.x), ex2(a1.y)),
                                     make_float2(__uint_as_float(v[jj + 2]),
                                                 __uint_as_float(v[jj + 3])));
        out[jj >> 1] = pack_bf16(e0.x, e0.y);
        out[(jj >> 1) + 1] = pack_bf16(e1.x, e1.y);
    }
}

// One 32-column block strictly below the diagonal block of row r: with p the
// block's last row, 2^(g_r - g_j) dt_j = 2^(g_r - g_p) * (2^(g_p - g_j) dt_j),
// both factors <= 1 (times dt), so the entries are cb[j] * u * vcol[j] with
// u = 2^(g_r - g_p) and vcol[j] = 2^(g_p - g_j) dt_j: no exponent per entry.
__device__ __forceinline__ void l_block_below(const uint32_t (&v)[32], int col0, float u,
                                              const float *vcol, uint32_t (&out)[16]) {
    const float2 u2 = make_float2(u, u);
#pragma unroll
    for (int jj = 0; jj < 32; jj += 4) {
        const float4 c4 = *reinterpret_cast<const float4 *>(vcol + col0 + jj);
        const float2 e0 = __fmul2_rn(
            __fmul2_rn(make_float2(__uint_as_float(v[jj]), __uint_as_float(v[jj + 1])),
                       make_float2(c4.x, c4.y)),
            u2);
        const float2 e1 = __fmul2_rn(
            __fmul2_rn(make_float2(__uint_as_float(v[jj + 2]), __uint_as_float(v[jj + 3])),
                       make_float2(c4.z, c4.w)),
            u2);
        out[jj >> 1] = pack_bf16(e0.x, e0.y);
        out[(jj >> 1) + 1] = pack_bf16(e1.x, e1.y);
    }
}

// Block-local cumulative sum of A dt over the 128 rows owned by one math
// warpgroup (thread r holds row r); returns g_r and g_end in log2 units.
// `bar` is the warpgroup's named barrier, `wsum` its 4-float scratch.
__device__ __forceinline__ void block_cumsum(float adt, int q, int lane, int bar, float *wsum,
                                             float &gr, float &gend) {
    float s = adt;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const float o = __shfl_up_sync(0xffffffffu, s, off);
        if (lane >= off) s += o;
    }
    if (lane == 31) wsum[q] = s;
    asm volatile("bar.sync %0, 128;" ::"r"(bar) : "memory");
    float pre = 0.f;
    for (int qq = 0; qq < q; ++qq) pre += wsum[qq];
    const float tot = ((wsum[0] + wsum[1]) + wsum[2]) + wsum[3];
    gr = (pre + s) * kLog2e;
    gend = tot * kLog2e;
}

// Warps: 0 = TMA producer; 1 = tensor-memory owner and MMA issuer; 2..9 =
// warpgroup A (w o x and the decay operand L; two warps per TMEM lane
// quarter, splitting the column blocks); 10..13 = warpgroup B (state update
// and y).  Block k uses stage s = k & 1 of every double buffer.  Tensor
// memory: [128 s, +128) = C B^T of stage s, then L in its first 64 columns
// and S^T in its last 64; [256 + 64 s, +64) = inter; [384 + 64 s, +64) = intra.
//
// Only the carried state is serial: h(k + 1) = 2^(g_end) h(k) + S(k), with S(k)
// independent of h.  The MMA issuer therefore polls its three inputs -- the
// state entering block k (for C h^T), the decay operand of block k (for L x
// and S^T) and the operands of block k + 1 (for C B^T) -- and issues
// whichever is ready, C h^T first.
__global__ void __launch_bounds__(kThreads, 1)
k_ssd_fused(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_b,
            const __grid_constant__ CUtensorMap tm_c, const __grid_constant__ CUtensorMap tm_y,
            const FusedParams p) {
    using SM = FusedSmem;
    constexpr uint32_t kCols = 512;
    constexpr uint32_t kIdCB = ptx::idesc_bf16_f32(128, 128, false, false);
    constexpr uint32_t kIdKmn = ptx::idesc_bf16_f32(128, 64, false, true);   // A K-major, B MN-major
    constexpr uint32_t kIdState = ptx::idesc_bf16_f32(128, 64, true, true);
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    float *grow_all = reinterpret_cast<float *>(smem + SM::kF);         // [2][128]
    float *ngd_all = grow_all + 256;                                     // [2][128]
    uint32_t *w2_all = reinterpret_cast<uint32_t *>(ngd_all + 256);      // [2][128]
    float *vcol_all = reinterpret_cast<float *>(w2_all + 256);           // [2][128]
    float *wsum_all = vcol_all + 256;                                    // [2][4]
    float *gpiv_all = wsum_all + 8;                                      // [2][4]
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + SM::kBar);
    uint64_t *full_C = bars, *full_B = bars + 2, *full_X = bars + 4, *cb_done = bars + 6,
             *inter_done = bars + 8, *L_ready = bars + 10, *is_done = bars + 12,
             *drain_done = bars + 14, *hb_ready = bars + 16;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 17);
    int *s_err = reinterpret_cast<int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // unit = (segment, batch, head), heads fastest so neighbouring CTAs share B, C in L2
    const int unit = blockIdx.x;
    const int h = unit % p.H;
    const int b = (unit / p.H) % p.B;
    const int seg = unit / (p.H * p.B);
    const int g = h / p.hpg;
    const int64_t t_begin = int64_t(seg) * p.seg_len;
    const int64_t t_end = t_begin + p.seg_len < p.L ? t_begin + p.seg_len : p.L;
    const int nblk = int((t_end - t_begin + 127) / 128);

    if (threadIdx.x == 0) {
        for (int s = 0; s < 2; ++s) {
            ptx::mbar_init(&full_C[s], 1);
            ptx::mbar_init(&full_B[s], 1);
            ptx::mbar_init(&full_X[s], 1);
            ptx::mbar_init(&cb_done[s], 1);
            ptx::mbar_init(&inter_done[s], 1);
            ptx::mbar_init(&L_ready[s], kWgA);
            ptx::mbar_init(&is_done[s], 1);
            ptx::mbar_init(&drain_done[s], 128);
        }
        ptx::mbar_init(hb_ready, 128);
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
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    bool ok = true;

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            for (int k = 0; k < nblk && ok; ++k) {
                const int s = k & 1, u = k >> 1;
                const uint32_t pp = (u - 1) & 1;  // phase of block k - 2 on this stage
                const int t0 = int(t_begin + int64_t(k) * 128);
                if (u > 0 && !ptx::mbar_wait(&inter_done[s], pp)) { ok = false; break; }
                ptx::mbar_arrive_expect_tx(&full_C[s], 32768);
                ptx::tma_load_4d(smem + SM::kC + s * 32768, &tm_c, &full_C[s], 0, g, t0, b);
                ptx::tma_load_4d(smem + SM::kC + s * 32768 + 16384, &tm_c, &full_C[s], 64, g, t0, b);
                if (u > 0 && !ptx::mbar_wait(&is_done[s], pp)) { ok = false; break; }
                ptx::mbar_arrive_expect_tx(&full_B[s], 32768);
                ptx::tma_load_4d(smem + SM::kB + s * 32768, &tm_b, &full_B[s], 0, g, t0, b);
                ptx::tma_load_4d(smem + SM::kB + s * 32768 + 16384, &tm_b, &full_B[s], 64, g, t0, b);
                if (u > 0 && !ptx::mbar_wait(&drain_done[s], pp)) { ok = false; break; }
                ptx::mbar_arrive_expect_tx(&full_X[s], 16384);
                ptx::tma_load_4d(smem + SM::kX + s * 16384, &tm_x, &full_X[s], 0, h, t0, b);
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
            int k_inter = 0, k_is = 0, k_cb = 0;   // next block of each product
            uint64_t idle_since = 0;
            while (k_inter < nblk || k_is < nblk) {
                bool progress = false;
                // C h^T(k): the state entering block k is in its operand tile
                if (k_inter < k_cb && ptx::mbar_test_wait(hb_ready, k_inter & 1)) {
                    const int s = k_inter & 1;
                    ptx::tc_fence_after();
                    const uint64_t c0 = dCk + uint64_t(s * 2048);
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks)   // MN-major operand: K step 16 rows = 2 KB
                        ptx::mma_bf16_ss(tmem + 256 + 64 * s, c0 + kKoff[ks],
                                         dHB + uint64_t(ks * 128), kIdKmn, ks != 0);
                    ptx::mma_commit(&inter_done[s]);
                    ++k_inter;
                    progress = true;
                }
                // L x(k) and S^T(k): block k's decay operand and w o x are ready and
                // its intra accumulator has been drained (block k - 2)
                if (k_is < k_cb) {
                    const int s = k_is & 1;
                    const uint32_t par = (k_is >> 1) & 1;
                    if (ptx::mbar_test_wait(&L_ready[s], par) &&
                        (k_is < 2 || ptx::mbar_test_wait(&drain_done[s], par ^ 1))) {
                        ptx::tc_fence_after();
                        const uint64_t x0 = dX + uint64_t(s * 1024);
                        const uint64_t xp0 = dXP + uint64_t(s * 1024);
                        const uint64_t bmn0 = dBmn + uint64_t(s * 2048);
                        const uint32_t t_cbl = tmem + 128 * s;
#pragma unroll
                        for (int ks = 0; ks < 8; ++ks)
                            ptx::mma_bf16_ts(tmem + 384 + 64 * s, t_cbl + ks * 8,
                                             x0 + uint64_t(ks * 128), kIdKmn, ks != 0);
#pragma unroll
                        for (int ks = 0; ks < 8; ++ks)
                            ptx::mma_bf16_ss(t_cbl + 64, bmn0 + uint64_t(ks * 128),
                                             xp0 + uint64_t(ks * 128), kIdState, ks != 0);
                        ptx::mma_commit(&is_done[s]);
                        ++k_is;
                        progress = true;
                    }
                }
                // C B^T(k): its operands landed and its stage's tensor memory is free:
                // L x and S^T of block k - 2 done, and S^T(k - 2) absorbed into the
                // state -- known once C h^T(k - 1) was issued, which waited for it
                if (k_cb < nblk && k_cb <= k_is + 1) {
                    const int s = k_cb & 1;
                    const uint32_t par = (k_cb >> 1) & 1;
                    if (ptx::mbar_test_wait(&full_C[s], par) && ptx::mbar_test_wait(&full_B[s], par) &&
                        (k_cb < 2 || (k_inter >= k_cb &&
                                      ptx::mbar_test_wait(&is_done[s], par ^ 1)))) {
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
            // every commit must land before tensor memory is released
            if (ok && !ptx::mbar_wait(&is_done[(nblk - 1) & 1], ((nblk - 1) >> 1) & 1)) ok = false;
            if (ok && !ptx::mbar_wait(&inter_done[(nblk - 1) & 1], ((nblk - 1) >> 1) & 1)) ok = false;
        }
    } else if (warp < 10) {
        // ---------------- warpgroup A: w o x and the decay operand ----------------
        const int q = warp & 3;
        const int half = (warp - 2) >> 2;          // which column blocks of the quarter
        const int r = 32 * q + lane;
        const int ta = threadIdx.x - 64;           // 0..255
        const uint32_t lane_off = uint32_t(32 * q) << 16;
        const float Ah = p.A[h];
        const float *dtp = p.dt + int64_t(b) * p.dt_sb + h;
        float dt_next = 0.f;
        if (half == 0) dt_next = (t_begin + r < t_end) ? __ldg(dtp + (t_begin + r) * p.dt_sl) : 0.f;
        for (int k = 0; k < nblk; ++k) {
            const int s = k & 1;
            const uint32_t par = (k >> 1) & 1;
            float *grow = grow_all + 128 * s;
            float *ngd = ngd_all + 128 * s;
            uint32_t *w2 = w2_all + 128 * s;
            float *vcol = vcol_all + 128 * s;
            float *gpiv = gpiv_all + 4 * s;
            if (half == 0) {
                const int64_t t = t_begin + int64_t(k) * 128 + r;
                const float dtr = dt_next;
                if (k + 1 < nblk) dt_next = (t + 128 < t_end) ? __ldg(dtp + (t + 128) * p.dt_sl) : 0.f;
                float gr, gend;
                block_cumsum(Ah * dtr, q, lane, 1, wsum_all, gr, gend);
                const float ngr = log2f(dtr) - gr;     // -inf for dt = 0
                grow[r] = gr;
                ngd[r] = ngr;
                const float w = ex2(gend - gr) * dtr;
                w2[r] = pack_bf16(w, w);
                // warp q holds column block q; its pivot is the block's last row
                const float gp = __shfl_sync(0xffffffffu, gr, 31);
                vcol[r] = ex2(gp + ngr);               // 2^(g_p - g_r) dt_r
                if (lane == 31) gpiv[q] = gp;
            }
            asm volatile("bar.sync 3, 256;" ::: "memory");
            const float gr = grow[r];

            // w o x into this stage's buffer (free once S(k - 2) has completed);
            // it does not need C B^T, so it runs while that product is computed
            if (!__all_sync(0xffffffffu,
                            ptx::mbar_wait(&full_X[s], par) &&
                                (k < 2 || ptx::mbar_wait(&is_done[s], par ^ 1)))) {
                ok = false;
                break;
            }
            {
                const uint4 *xs = reinterpret_cast<const uint4 *>(smem + SM::kX + s * 16384);
                uint4 *xp = reinterpret_cast<uint4 *>(smem + SM::kXP + s * 16384);
#pragma unroll
                for (int rr = 0; rr < 4; ++rr) {
                    const int chunk = ta + kWgA * rr;    // 16-byte chunk; row j = chunk / 8
                    const uint32_t wv = w2[chunk >> 3];
                    const __nv_bfloat162 wb = *reinterpret_cast<const __nv_bfloat162 *>(&wv);
                    uint4 v = xs[chunk];
                    __nv_bfloat162 *v2 = reinterpret_cast<__nv_bfloat162 *>(&v);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) v2[kk] = __hmul2(v2[kk], wb);
                    xp[chunk] = v;
                }
            }
            ptx::fence_proxy_async_smem();

            // L, in place over C B^T: this warp owns column blocks half and
            // half + 2 of its rows (blocks past the diagonal block q are zero).
            // Every read of the stage's C B^T completes before any write.
            if (!__all_sync(0xffffffffu, ptx::mbar_wait(&cb_done[s], par))) { ok = false; break; }
            ptx::tc_fence_after();
            {
                const uint32_t tL = tmem + 128 * s + lane_off;
                const int c0 = half, c1 = half + 2;
                uint32_t v0[32], v1[32], out[16];
                if (c0 <= q) ptx::tmem_ld32(tL + 32 * c0, v0);
                if (c1 <= q) ptx::tmem_ld32(tL + 32 * c1, v1);
                ptx::tmem_ld_wait();
                ptx::tc_fence_before();
                asm volatile("bar.sync 3, 256;" ::: "memory");
                ptx::tc_fence_after();
                if (c0 <= q) {
                    if (c0 == q) l_block(v0, 32 * c0, true, r, gr, ngd, out);
                    else l_block_below(v0, 32 * c0, ex2(gr - gpiv[c0]), vcol, out);
                } else {
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) out[jj] = 0u;
                }
                ptx::tmem_st16(tL + 16 * c0, out);
                if (c1 <= q) {
                    if (c1 == q) l_block(v1, 32 * c1, true, r, gr, ngd, out);
                    else l_block_below(v1, 32 * c1, ex2(gr - gpiv[c1]), vcol, out);
                } else {
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) out[jj] = 0u;
                }
                ptx::tmem_st16(tL + 16 * c1, out);
                ptx::tmem_st_wait();
            }
            ptx::tc_fence_before();
            ptx::mbar_arrive(&L_ready[s]);
        }
    } else {
        // ---------------- warpgroup B: carried state and y ----------------
        const int q = warp & 3;
        const int r = 32 * q + lane;
        const uint32_t lane_off = uint32_t(32 * q) << 16;
        const float Ah = p.A[h];
        const float Dh = p.D ? p.D[h] : 0.f;
        const float2 D2 = make_float2(Dh, Dh);
        uint8_t *hb = smem + SM::kHB;
        const size_t slab = size_t(b) * p.H + h;
        float2 hreg[32];   // state row n = r, headdim pairs (2m, 2m + 1), fp32
        const float *hin = p.h_in ? p.h_in + (size_t(seg) * p.B * p.H + slab) * 8192 : nullptr;
#pragma unroll
        for (int m = 0; m < 32; ++m)
            hreg[m] = hin ? make_float2(hin[(2 * m) * 128 + r], hin[(2 * m + 1) * 128 + r])
                          : make_float2(0.f, 0.f);
        write_state_row(hb, r, hreg);
        ptx::fence_proxy_async_smem();
        ptx::mbar_arrive(hb_ready);

        const float *dtp = p.dt + int64_t(b) * p.dt_sb + h;
        float dt_next = (t_begin + r < t_end) ? __ldg(dtp + (t_begin + r) * p.dt_sl) : 0.f;
        for (int k = 0; k < nblk; ++k) {
            const int s = k & 1;
            const uint32_t par = (k >> 1) & 1;
            const int64_t t = t_begin + int64_t(k) * 128 + r;
            const float dtr = dt_next;
            if (k + 1 < nblk) dt_next = (t + 128 < t_end) ? __ldg(dtp + (t + 128) * p.dt_sl) : 0.f;
            float gr, gend;
            block_cumsum(Ah * dtr, q, lane, 2, wsum_all + 4, gr, gend);
            asm volatile("bar.sync 2, 128;" ::: "memory");   // wsum reads done before reuse

            // state: h(k + 1) = 2^(g_end) h(k) + S(k); its bf16 copy feeds C h^T(k + 1)
            // once C h^T(k) has read the current one
            if (!__all_sync(0xffffffffu, ptx::mbar_wait(&is_done[s], par) &&
                                             ptx::mbar_wait(&inter_done[s], par))) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            {
                const float dend = ex2(gend);
                const float2 d2 = make_float2(dend, dend);
#pragma unroll
                for (int cb = 0; cb < 2; ++cb) {
                    uint32_t sv[32];
                    ptx::tmem_ld32(tmem + 128 * s + 64 + lane_off + 32 * cb, sv);
                    ptx::tmem_ld_wait();
#pragma unroll
                    for (int m = 0; m < 16; ++m)
                        hreg[16 * cb + m] =
                            __ffma2_rn(d2, hreg[16 * cb + m],
                                       make_float2(__uint_as_float(sv[2 * m]),
                                                   __uint_as_float(sv[2 * m + 1])));
                }
                write_state_row(hb, r, hreg);
            }
            ptx::fence_proxy_async_smem();
            ptx::tc_fence_before();
            ptx::mbar_arrive(hb_ready);

            // y(k) = 2^(g_i) inter + intra + D x, written over this block's x tile
            // (each thread reads its x row before writing its y row there), then
            // stored as one tile by TMA (rows past the sequence end are clipped)
            {
                const float e_i = ex2(gr);
                const float2 e2 = make_float2(e_i, e_i);
                uint8_t *tile = smem + SM::kX + s * 16384;
                uint8_t *row = tile + r * 128;
#pragma unroll 1
                for (int cb = 0; cb < 4; ++cb) {
                    uint32_t a[16], d[16];
                    ptx::tmem_ld16(tmem + 256 + 64 * s + lane_off + 16 * cb, a);
                    ptx::tmem_ld16(tmem + 384 + 64 * s + lane_off + 16 * cb, d);
                    ptx::tmem_ld_wait();
#pragma unroll
                    for (int c4 = 0; c4 < 2; ++c4) {
                        const int ch = 2 * cb + c4;
                        uint4 *cp = reinterpret_cast<uint4 *>(row + ((ch ^ (r & 7)) << 4));
                        const uint4 xv = *cp;
                        const uint32_t *xu = reinterpret_cast<const uint32_t *>(&xv);
                        uint32_t o[4];
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            const int jj = 8 * c4 + 2 * kk;
                            float2 acc = __ffma2_rn(
                                make_float2(__uint_as_float(a[jj]), __uint_as_float(a[jj + 1])), e2,
                                make_float2(__uint_as_float(d[jj]), __uint_as_float(d[jj + 1])));
                            acc = __ffma2_rn(unpack_bf16(xu[kk]), D2, acc);
                            o[kk] = pack_bf16(acc.x, acc.y);
                        }
                        *cp = make_uint4(o[0], o[1], o[2], o[3]);
                    }
                }
                ptx::fence_proxy_async_smem();
                asm volatile("bar.sync 2, 128;" ::: "memory");
                if (warp == 10 && lane == 0) {
                    ptx::tma_store_4d(&tm_y, tile, 0, h, int(t_begin + int64_t(k) * 128), b);
                    ptx::bulk_commit_group();
                    ptx::bulk_wait_group_read0();   // the tile is reloaded after drain_done
                }
            }
            ptx::tc_fence_before();
            ptx::mbar_arrive(&drain_done[s]);
        }
        if (warp == 10 && lane == 0) ptx::bulk_wait_group0();
        if (ok && p.h_out) {
            float *ho = p.h_out + slab * 8192;
#pragma unroll
            for (int m = 0; m < 32; ++m) {
                ho[(2 * m) * 128 + r] = hreg[m].x;
                ho[(2 * m + 1) * 128 + r] = hreg[m].y;
            }
        }
    }
    if (!ok) atomicOr(s_err, 1);
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, kCols);
    }
    if (threadIdx.x == 0 && *s_err) atomicOr(p.err, 1u);
}

}  // namespace

bool fused_supported(const Dims &d, int xdt) {
    return xdt == DT_BF16 && d.P == 64 && d.N == 128 && d.Q % 128 == 0;
}

cudaError_t launch_fused(const Args &a, cudaStream_t s) {
    const Dims &d = a.d;
    CUtensorMap tm_x, tm_b, tm_c;
    const uint32_t box[4] = {64, 1, 128, 1};
    const uint64_t xd[4] = {64, uint64_t(d.H), uint64_t(d.L), uint64_t(d.B)};
    const uint64_t xs[3] = {uint64_t(a.x_sh) * 2, uint64_t(a.x_sl) * 2, uint64_t(a.x_sb) * 2};
    const uint64_t bd[4] = {128, uint64_t(d.G), uint64_t(d.L), uint64_t(d.B)};
    const uint64_t bs[3] = {uint64_t(a.b_sg) * 2, uint64_t(a.b_sl) * 2, uint64_t(a.b_sb) * 2};
    const uint64_t cs[3] = {uint64_t(a.c_sg) * 2, uint64_t(a.c_sl) * 2, uint64_t(a.c_sb) * 2};
    cudaError_t e = make_tmap_bf16(&tm_x, a.x, 4, xd, xs, box);
    if (e != cudaSuccess) return e;
    if ((e = make_tmap_bf16(&tm_b, a.Bm, 4, bd, bs, box)) != cudaSuccess) return e;
    if ((e = make_tmap_bf16(&tm_c, a.Cm, 4, bd, cs, box)) != cudaSuccess) return e;
    CUtensorMap tm_y;
    const uint64_t ys[3] = {uint64_t(a.y_sh) * 2, uint64_t(a.y_sl) * 2, uint64_t(a.y_sb) * 2};
    if ((e = make_tmap_bf16(&tm_y, a.y, 4, xd, ys, box)) != cudaSuccess) return e;
    unsigned int *err = nullptr;
    if ((e = device_error_word(&err)) != cudaSuccess) return e;
    FusedParams p{};
    p.L = d.L;
    p.seg_len = ((d.L + 127) / 128) * 128;
    p.B = int(d.B);
    p.H = int(d.H);
    p.hpg = int(d.hpg());
    p.nseg = 1;
    p.dt = a.dt;
    p.dt_sb = a.dt_sb;
    p.dt_sl = a.dt_sl;
    p.A = a.A;
    p.D = a.D;
    p.h_in = a.h0;
    p.h_out = a.final_states;
    p.y = static_cast<__nv_bfloat16 *>(a.y);
    p.y_sb = a.y_sb;
    p.y_sl = a.y_sl;
    p.y_sh = a.y_sh;
    p.err = err;
    const int smem = FusedSmem::kBytes;
    e = cudaFuncSetAttribute(k_ssd_fused, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const unsigned units = unsigned(d.B * d.H) * unsigned(p.nseg);
    k_ssd_fused<<<units, kThreads, smem, s>>>(tm_x, tm_b, tm_c, tm_y, p);
    return cudaGetLastError();
}

}  // namespace ssd
