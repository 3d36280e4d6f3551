// Tensor-core (tcgen05 + TMA) chunk_state and chunk_scan for fp32 inputs,
// P = 64, N = 128, Q of 128 or 256.
//
// The tensor cores take bf16 operands here; an fp32 operand a is carried as
// the pair a_hi = bf16(a), a_lo = bf16(a - a_hi), whose sum is a to ~2^-17
// relative, and each product is formed from three MMAs,
//     a b ~ a_hi b_hi + a_hi b_lo + a_lo b_hi,
// dropping a_lo b_lo (~2^-16 relative), with fp32 accumulation.  The
// products are those of "Accelerating Mamba-2 with High-Performance Forward
// Pass Kernels in NVIDIA CUDA Tile" ("Kernel 2: fwd_pass_state" without the
// carried state; "Kernel 3: compute_out"), as in the bf16 kernels of
// ssd_tc.cu; every elementwise factor (w_j = 2^(G_last - G_j) dt_j, the
// decay operand L, the scale 2^(G_i), D x) is applied in fp32 before a split
// or after the accumulators are read.
//
// The inputs x, B, C and the chunk-entering states h_prev are split once
// into contiguous bf16 hi / lo tensors in the workspace (k_split_hilo), so the
// kernels load them with the bf16 tensor maps and 128-byte swizzled layouts
// of the bf16 kernels.
#include "ptx_sm100.cuh"
#include "ssd_internal.h"
#include "ssd_tc.cuh"
#define SSD_DBG_FILE 6u   // kDbgTcF32
#include "ssd_debug.cuh"
#include "ssd_tmap.h"

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace ssd {
namespace {

constexpr int kTile = 8192;  // one 64-row x 128-byte swizzled tile (bf16 64 x 64)

__device__ __forceinline__ uint8_t *align1024(uint8_t *p) {
    return reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// hi = bf16(v), lo = bf16(v - hi), for two values, packed as bf16x2.
__device__ __forceinline__ void split2(float v0, float v1, uint32_t &hi, uint32_t &lo) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(v0, v1);
    const float2 hf = __bfloat1622float2(h);
    const __nv_bfloat162 l = __floats2bfloat162_rn(v0 - hf.x, v1 - hf.y);
    hi = *reinterpret_cast<const uint32_t *>(&h);
    lo = *reinterpret_cast<const uint32_t *>(&l);
}

// The fp32 value of one bf16x2 word of hi plus the matching word of lo.
__device__ __forceinline__ float2 join2(uint32_t hi, uint32_t lo) {
    const float2 h = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&hi));
    const float2 l = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&lo));
    return make_float2(h.x + l.x, h.y + l.y);
}

// src [n0][n1][n2][inner] fp32 with element strides (s0, s1, s2, 1) ->
// contiguous bf16 hi, lo of the same shape.
__global__ void __launch_bounds__(256)
k_split_hilo(const float *src, int64_t n1, int64_t n2, int64_t inner, int64_t s0, int64_t s1,
             int64_t s2, int64_t total, __nv_bfloat16 *hi, __nv_bfloat16 *lo, unsigned int *err,
             int64_t n_src) {
    const int64_t stride = int64_t(gridDim.x) * blockDim.x;
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += stride) {
        int64_t r = i;
        const int64_t c = r % inner;
        r /= inner;
        const int64_t i2 = r % n2;
        r /= n2;
        const int64_t i1 = r % n1, i0 = r / n1;
        const int64_t o = i0 * s0 + i1 * s1 + i2 * s2 + c;
        const float v = SSD_IDX_OK(err, o, n_src) ? src[o] : 0.f;
        const __nv_bfloat16 h = __float2bfloat16_rn(v);
        hi[i] = h;
        lo[i] = __float2bfloat16_rn(v - __bfloat162float(h));
    }
}

// ---------------------------------------------------------------------------
// chunk_state:  S_c^T [n][p] = sum_j B_j[n] (w_j x_j[p]),  w_j = 2^(G_last - G_j) dt_j.
// One CTA per (chunk, KH heads of one group, batch).  Tokens stream through
// shared memory 64 at a time: B_hi, B_lo (two tiles each), x_hi, x_lo (one
// tile per head each).  Four math warps form w_j x_j = w_j (x_hi + x_lo) in
// fp32 and write its hi / lo split back over x_hi / x_lo; one thread issues
// the three MMAs per 16-token step with B^T as the M = 128 operand.

struct StateF32Params {
    int64_t L, Lp;
    int H, hpg, Q;
    const float *dt;
    int64_t dt_sb, dt_sl;
    const float *G;
    float *S;
    int64_t nc;
    unsigned int *err;
    int64_t n_dt, n_G, n_S;   // element extents (debug build)
};

template <int KH, int NSTG>
struct StateF32Smem {
    static constexpr int kStageBytes = (4 + 2 * KH) * kTile;   // B hi, lo; x hi, lo per head
    static constexpr int kStages = NSTG * kStageBytes;
    static constexpr int kBytes = kStages + KH * 256 * 4 + 256 + 1024;
};

template <int KH, int NSTG>
__global__ void __launch_bounds__(192, 1)
k_chunk_state_tc_f32(const __grid_constant__ CUtensorMap tm_xh, const __grid_constant__ CUtensorMap tm_xl,
                     const __grid_constant__ CUtensorMap tm_bh, const __grid_constant__ CUtensorMap tm_bl,
                     const StateF32Params p) {
    using SM = StateF32Smem<KH, NSTG>;
    constexpr uint32_t kCols = KH * 64;
    constexpr uint32_t kIdesc = ptx::idesc_bf16_f32(128, 64, true, true);
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    float *wts = reinterpret_cast<float *>(smem + SM::kStages);   // [KH][Q]
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + SM::kStages + KH * 256 * 4);
    uint64_t *full = bars, *scaled = bars + NSTG, *empty = bars + 2 * NSTG,
             *accfull = bars + 3 * NSTG;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 3 * NSTG + 1);
    int *s_err = reinterpret_cast<int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t c = blockIdx.x, b = blockIdx.z;
    const int h0 = blockIdx.y * KH;
    const int g = h0 / p.hpg;
    const int Q = p.Q, nkb = Q / 64;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NSTG; ++s) {
            ptx::mbar_init(&full[s], 1);
            ptx::mbar_init(&scaled[s], 128);
            ptx::mbar_init(&empty[s], 1);
        }
        ptx::mbar_init(accfull, 1);
        *s_err = 0;
        ptx::fence_mbar_init();
        ptx::prefetch_tmap(&tm_xh);
        ptx::prefetch_tmap(&tm_xl);
        ptx::prefetch_tmap(&tm_bh);
        ptx::prefetch_tmap(&tm_bl);
    }
    if (warp == 1) {
        ptx::tmem_alloc(tmem_slot, kCols);
        ptx::tmem_relinquish();
    }
    if (warp >= 2) {
        // per-token weights w_j = 2^(G_last - G_j) dt_j (0 past the sequence end)
        for (int e = threadIdx.x - 64; e < KH * Q; e += 128) {
            const int i = e / Q, j = e - i * Q;
            const int64_t gb = (b * p.H + h0 + i) * p.Lp + c * Q;
            const int64_t t = c * Q + j;
            const int64_t dto = b * p.dt_sb + t * p.dt_sl + h0 + i;
            wts[e] = (t < p.L && SSD_IDX_OK(p.err, gb + Q - 1, p.n_G) &&
                      SSD_IDX_OK(p.err, dto, p.n_dt))
                         ? exp2f(p.G[gb + Q - 1] - p.G[gb + j]) * __ldg(p.dt + dto)
                         : 0.f;
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    bool ok = true;

    if (warp == 0) {
        if (lane == 0) {
            for (int kb = 0; kb < nkb && ok; ++kb) {
                const int s = kb % NSTG, u = kb / NSTG;
                if (u > 0 && !ptx::mbar_wait(&empty[s], (u - 1) & 1)) {
                    ok = false;
                    break;
                }
                uint8_t *st = smem + s * SM::kStageBytes;
                ptx::mbar_arrive_expect_tx(&full[s], SM::kStageBytes);
                const int t0 = int(c * Q + kb * 64);
                ptx::tma_load_4d(st, &tm_bh, &full[s], 0, g, t0, int(b));
                ptx::tma_load_4d(st + kTile, &tm_bh, &full[s], 64, g, t0, int(b));
                ptx::tma_load_4d(st + 2 * kTile, &tm_bl, &full[s], 0, g, t0, int(b));
                ptx::tma_load_4d(st + 3 * kTile, &tm_bl, &full[s], 64, g, t0, int(b));
                for (int i = 0; i < KH; ++i) {
                    ptx::tma_load_4d(st + (4 + i) * kTile, &tm_xh, &full[s], 0, h0 + i, t0, int(b));
                    ptx::tma_load_4d(st + (4 + KH + i) * kTile, &tm_xl, &full[s], 0, h0 + i, t0,
                                     int(b));
                }
            }
            // never leave the CTA with copies in flight
            for (int kb = (nkb > NSTG ? nkb - NSTG : 0); kb < nkb; ++kb)
                if (!ptx::mbar_wait(&full[kb % NSTG], (kb / NSTG) & 1, 200000000ull)) ok = false;
        }
    } else if (warp == 1) {
        if (lane == 0) {
            for (int kb = 0; kb < nkb && ok; ++kb) {
                const int s = kb % NSTG, u = kb / NSTG;
                if (!ptx::mbar_wait(&scaled[s], u & 1)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t sb = ptx::smem_u32(smem + s * SM::kStageBytes);
#pragma unroll
                for (int i = 0; i < KH; ++i) {
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        // A = B^T: M = state (two 64-wide atoms 8 KB apart), K = tokens
                        const uint64_t a_hi = ptx::sdesc(sb + k * 2048, kTile, 1024);
                        const uint64_t a_lo = ptx::sdesc(sb + 2 * kTile + k * 2048, kTile, 1024);
                        // B = w x of head i: N = headdim (one atom), K = tokens
                        const uint64_t b_hi = ptx::sdesc(sb + (4 + i) * kTile + k * 2048, kTile, 1024);
                        const uint64_t b_lo =
                            ptx::sdesc(sb + (4 + KH + i) * kTile + k * 2048, kTile, 1024);
                        ptx::mma_bf16_ss(tmem + i * 64, a_hi, b_hi, kIdesc, (kb | k) != 0);
                        ptx::mma_bf16_ss(tmem + i * 64, a_hi, b_lo, kIdesc, 1);
                        ptx::mma_bf16_ss(tmem + i * 64, a_lo, b_hi, kIdesc, 1);
                    }
                }
                ptx::mma_commit(&empty[s]);
            }
            ptx::mma_commit(accfull);
            if (!ptx::mbar_wait(accfull, 0)) ok = false;
        }
    } else {
        const int mt = threadIdx.x - 64;   // 0..127
        for (int kb = 0; kb < nkb; ++kb) {
            const int s = kb % NSTG, u = kb / NSTG;
            if (!ptx::mbar_wait(&full[s], u & 1)) {
                ok = false;
                break;
            }
            uint8_t *st = smem + s * SM::kStageBytes;
#pragma unroll
            for (int i = 0; i < KH; ++i) {
                uint4 *xh = reinterpret_cast<uint4 *>(st + (4 + i) * kTile);
                uint4 *xl = reinterpret_cast<uint4 *>(st + (4 + KH + i) * kTile);
                const float *w = wts + i * Q + kb * 64;
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const int chunk = mt + 128 * r;   // 16-byte chunk; 8 per 128-byte row
                    const float wj = w[chunk >> 3];
                    uint4 vh = xh[chunk], vl = xl[chunk];
                    uint32_t *uh = reinterpret_cast<uint32_t *>(&vh);
                    uint32_t *ul = reinterpret_cast<uint32_t *>(&vl);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float2 xv = join2(uh[q], ul[q]);
                        split2(xv.x * wj, xv.y * wj, uh[q], ul[q]);
                    }
                    xh[chunk] = vh;
                    xl[chunk] = vl;
                }
            }
            ptx::fence_proxy_async_smem();
            ptx::mbar_arrive(&scaled[s]);
        }
        const bool go = __all_sync(0xffffffffu, ok && ptx::mbar_wait(accfull, 0));
        if (go) {
            ptx::tc_fence_after();
            const int q = warp & 3;
            const int n = 32 * q + lane;
            const uint32_t row = tmem + (uint32_t(32 * q) << 16);
#pragma unroll
            for (int i = 0; i < KH; ++i) {
                const int64_t so = ((b * p.nc + c) * p.H + h0 + i) * (64 * 128);
                if (!SSD_IDX_OK(p.err, so + 64 * 128 - 1, p.n_S)) continue;
                float *S = p.S + so + n;
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    uint32_t r[16];
                    ptx::tmem_ld16(row + i * 64 + cc * 16, r);
                    ptx::tmem_ld_wait();
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) S[(cc * 16 + jj) * 128] = __uint_as_float(r[jj]);
                }
            }
        } else {
            ok = false;
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

// ---------------------------------------------------------------------------
// chunk_scan ("Kernel 3: compute_out"): one CTA per (128-row block r of chunk
// c, head h, batch b):
//     y_i = 2^G_i (C_i h_prev^T) + sum_{s<=r} sum_j L_ij x_j + D x_i,
//     L_ij = [j <= i] (C_i . B_j) 2^(G_i - G_j) dt_j,
// in fp32 out.  The column blocks s = 0 .. r are taken one after another:
// B(s) hi / lo land, C B^T(s) is formed in tensor memory, the four math warps
// turn it into L(s) in fp32 and write its hi / lo split over B(s)'s tiles,
// and L(s) x(s) accumulates; the next block's B and x are loaded once that
// product has completed.  The last x loaded is x(r), which the epilogue
// reads for D x.

struct ScanF32Params {
    int64_t L, Lp, nc;
    int H, hpg, Q;
    const float *dt;
    int64_t dt_sb, dt_sl;
    const float *G;
    const float *D;
    float *y;
    int64_t y_sb, y_sl, y_sh;
    unsigned int *err;
    int64_t n_dt, n_G, n_y;   // element extents (debug build)
};

struct ScanF32Smem {
    static constexpr int kC = 0;            // C hi, lo: 2 x [128][128 B] each
    static constexpr int kHP = 65536;       // h_prev hi, lo: 2 x [64][128 B] each
    static constexpr int kB = 98304;        // B(s) hi, lo: 2 x [128][128 B] each; then L(s) hi, lo
    static constexpr int kX = 163840;       // x(s) hi, lo: [128][128 B] each
    static constexpr int kF = 196608;       // floats: gi[128], gj[2 * 128], dtj[2 * 128]
    static constexpr int kBar = kF + (128 + 4 * 128) * 4;
    static constexpr int kBytes = kBar + 256 + 1024;
};
static_assert(ScanF32Smem::kBytes <= 232448, "shared memory above the per-CTA limit");

__global__ void __launch_bounds__(192, 1)
k_chunk_scan_tc_f32(const __grid_constant__ CUtensorMap tm_xh, const __grid_constant__ CUtensorMap tm_xl,
                    const __grid_constant__ CUtensorMap tm_bh, const __grid_constant__ CUtensorMap tm_bl,
                    const __grid_constant__ CUtensorMap tm_ch, const __grid_constant__ CUtensorMap tm_cl,
                    const __grid_constant__ CUtensorMap tm_hh, const __grid_constant__ CUtensorMap tm_hl,
                    const ScanF32Params p) {
    using SM = ScanF32Smem;
    constexpr uint32_t kCols = 256;   // C B^T [0, 128), inter [128, 192), intra [192, 256)
    constexpr uint32_t kIdCB = ptx::idesc_bf16_f32(128, 128, false, false);
    constexpr uint32_t kIdInter = ptx::idesc_bf16_f32(128, 64, false, false);
    constexpr uint32_t kIdIntra = ptx::idesc_bf16_f32(128, 64, false, true);
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    float *gi = reinterpret_cast<float *>(smem + SM::kF);
    float *gj = gi + 128;
    float *dtj = gj + 2 * 128;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + SM::kBar);
    uint64_t *bar_in0 = bars, *bar_in = bars + 1, *bar_cb = bars + 2, *bar_L = bars + 3,
             *bar_free = bars + 4, *bar_acc = bars + 5;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 6);
    int *s_err = reinterpret_cast<int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int QB = p.Q / 128;
    const int64_t c = blockIdx.x / QB;
    const int r = int(blockIdx.x % QB);
    const int h = blockIdx.y;
    const int64_t b = blockIdx.z;
    const int g = h / p.hpg;
    const int Q = p.Q;
    const int nblk = r + 1;

    if (threadIdx.x == 0) {
        ptx::mbar_init(bar_in0, 1);
        ptx::mbar_init(bar_in, 1);
        ptx::mbar_init(bar_cb, 1);
        ptx::mbar_init(bar_L, 128);
        ptx::mbar_init(bar_free, 1);
        ptx::mbar_init(bar_acc, 1);
        *s_err = 0;
        ptx::fence_mbar_init();
        ptx::prefetch_tmap(&tm_xh);
        ptx::prefetch_tmap(&tm_xl);
        ptx::prefetch_tmap(&tm_bh);
        ptx::prefetch_tmap(&tm_bl);
        ptx::prefetch_tmap(&tm_ch);
        ptx::prefetch_tmap(&tm_cl);
        ptx::prefetch_tmap(&tm_hh);
        ptx::prefetch_tmap(&tm_hl);
    }
    if (warp == 1) {
        ptx::tmem_alloc(tmem_slot, kCols);
        ptx::tmem_relinquish();
    }
    if (warp >= 2) {
        const int i = threadIdx.x - 64;
        const int64_t gb = (b * p.H + h) * p.Lp + c * Q;
        gi[i] = SSD_IDX_OK(p.err, gb + r * 128 + i, p.n_G) ? p.G[gb + r * 128 + i] : 0.f;
        for (int s = 0; s < nblk; ++s) {
            const int64_t t = c * Q + s * 128 + i;
            const int64_t dto = b * p.dt_sb + t * p.dt_sl + h;
            gj[s * 128 + i] = SSD_IDX_OK(p.err, gb + s * 128 + i, p.n_G) ? p.G[gb + s * 128 + i] : 0.f;
            dtj[s * 128 + i] = (t < p.L && SSD_IDX_OK(p.err, dto, p.n_dt)) ? __ldg(p.dt + dto) : 0.f;
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t t_inter = tmem + 128, t_intra = tmem + 192;
    bool ok = true;

    if (warp == 0) {
        if (lane == 0) {
            const int t_r = int(c * Q + r * 128);
            const int hp_row = int(((b * p.nc + c) * p.H + h) * 64);
            ptx::mbar_arrive_expect_tx(bar_in0, 2 * 32768 + 2 * 16384);
            ptx::tma_load_4d(smem + SM::kC, &tm_ch, bar_in0, 0, g, t_r, int(b));
            ptx::tma_load_4d(smem + SM::kC + 16384, &tm_ch, bar_in0, 64, g, t_r, int(b));
            ptx::tma_load_4d(smem + SM::kC + 32768, &tm_cl, bar_in0, 0, g, t_r, int(b));
            ptx::tma_load_4d(smem + SM::kC + 49152, &tm_cl, bar_in0, 64, g, t_r, int(b));
            ptx::tma_load_3d(smem + SM::kHP, &tm_hh, bar_in0, 0, hp_row, 0);
            ptx::tma_load_3d(smem + SM::kHP + 8192, &tm_hh, bar_in0, 64, hp_row, 0);
            ptx::tma_load_3d(smem + SM::kHP + 16384, &tm_hl, bar_in0, 0, hp_row, 0);
            ptx::tma_load_3d(smem + SM::kHP + 24576, &tm_hl, bar_in0, 64, hp_row, 0);
            for (int s = 0; s < nblk; ++s) {
                // B(s), x(s) go where L(s - 1) x(s - 1) has finished reading
                if (s > 0 && !ptx::mbar_wait(bar_free, (s - 1) & 1)) {
                    ok = false;
                    break;
                }
                const int t_s = int(c * Q + s * 128);
                ptx::mbar_arrive_expect_tx(bar_in, 2 * 32768 + 2 * 16384);
                ptx::tma_load_4d(smem + SM::kB, &tm_bh, bar_in, 0, g, t_s, int(b));
                ptx::tma_load_4d(smem + SM::kB + 16384, &tm_bh, bar_in, 64, g, t_s, int(b));
                ptx::tma_load_4d(smem + SM::kB + 32768, &tm_bl, bar_in, 0, g, t_s, int(b));
                ptx::tma_load_4d(smem + SM::kB + 49152, &tm_bl, bar_in, 64, g, t_s, int(b));
                ptx::tma_load_4d(smem + SM::kX, &tm_xh, bar_in, 0, h, t_s, int(b));
                ptx::tma_load_4d(smem + SM::kX + 16384, &tm_xl, bar_in, 0, h, t_s, int(b));
            }
            // never leave the CTA with copies in flight
            if (!ptx::mbar_wait(bar_in0, 0, 200000000ull)) ok = false;
            if (ok && !ptx::mbar_wait(bar_in, (nblk - 1) & 1, 200000000ull)) ok = false;
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t sC = ptx::smem_u32(smem + SM::kC);
            const uint32_t sB = ptx::smem_u32(smem + SM::kB);
            const uint32_t sX = ptx::smem_u32(smem + SM::kX);
            ok = ptx::mbar_wait(bar_in0, 0);
            for (int s = 0; s < nblk && ok; ++s) {
                if (!ptx::mbar_wait(bar_in, s & 1)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                // C B^T(s) = C_hi B_hi^T + C_hi B_lo^T + C_lo B_hi^T
#pragma unroll
                for (int kb = 0; kb < 2; ++kb)
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const uint64_t ch = ptx::sdesc(sC + kb * 16384 + k * 32, 16, 1024);
                        const uint64_t cl = ptx::sdesc(sC + 32768 + kb * 16384 + k * 32, 16, 1024);
                        const uint64_t bh = ptx::sdesc(sB + kb * 16384 + k * 32, 16, 1024);
                        const uint64_t bl = ptx::sdesc(sB + 32768 + kb * 16384 + k * 32, 16, 1024);
                        ptx::mma_bf16_ss(tmem, ch, bh, kIdCB, (kb | k) != 0);
                        ptx::mma_bf16_ss(tmem, ch, bl, kIdCB, 1);
                        ptx::mma_bf16_ss(tmem, cl, bh, kIdCB, 1);
                    }
                ptx::mma_commit(bar_cb);
                if (s == 0) {
                    // inter = C h_prev^T, the same three products
                    const uint32_t sH = ptx::smem_u32(smem + SM::kHP);
#pragma unroll
                    for (int kb = 0; kb < 2; ++kb)
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const uint64_t ch = ptx::sdesc(sC + kb * 16384 + k * 32, 16, 1024);
                            const uint64_t cl =
                                ptx::sdesc(sC + 32768 + kb * 16384 + k * 32, 16, 1024);
                            const uint64_t hh = ptx::sdesc(sH + kb * 8192 + k * 32, 16, 1024);
                            const uint64_t hl = ptx::sdesc(sH + 16384 + kb * 8192 + k * 32, 16, 1024);
                            ptx::mma_bf16_ss(t_inter, ch, hh, kIdInter, (kb | k) != 0);
                            ptx::mma_bf16_ss(t_inter, ch, hl, kIdInter, 1);
                            ptx::mma_bf16_ss(t_inter, cl, hh, kIdInter, 1);
                        }
                }
                if (!ptx::mbar_wait(bar_L, s & 1)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                // L(s) x(s) = L_hi x_hi + L_hi x_lo + L_lo x_hi (L over B's tiles)
#pragma unroll
                for (int kb = 0; kb < 2; ++kb)
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const uint64_t lh = ptx::sdesc(sB + kb * 16384 + k * 32, 16, 1024);
                        const uint64_t ll = ptx::sdesc(sB + 32768 + kb * 16384 + k * 32, 16, 1024);
                        const uint64_t xh = ptx::sdesc(sX + (kb * 4 + k) * 2048, 16384, 1024);
                        const uint64_t xl = ptx::sdesc(sX + 16384 + (kb * 4 + k) * 2048, 16384, 1024);
                        ptx::mma_bf16_ss(t_intra, lh, xh, kIdIntra, (s | kb | k) != 0);
                        ptx::mma_bf16_ss(t_intra, lh, xl, kIdIntra, 1);
                        ptx::mma_bf16_ss(t_intra, ll, xh, kIdIntra, 1);
                    }
                ptx::mma_commit(bar_free);
            }
            ptx::mma_commit(bar_acc);
            if (!ptx::mbar_wait(bar_acc, 0)) ok = false;
        }
    } else {
        // tile row owned by this thread = the TMEM lane it may access: warp w
        // reaches lanes 32 (w % 4) .. 32 (w % 4) + 31
        const int i = 32 * (warp & 3) + lane;
        const uint32_t lane_off = uint32_t(32 * (warp & 3)) << 16;
        const float g_i = gi[i];
        for (int s = 0; s < nblk; ++s) {
            const bool go = __all_sync(0xffffffffu, ptx::mbar_wait(bar_cb, s & 1));
            if (!go) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            uint8_t *Lh = smem + SM::kB + i * 128;
            uint8_t *Ll = Lh + 32768;
            const bool diag = (s == r);
#pragma unroll 1
            for (int cb = 0; cb < 4; ++cb) {
                uint32_t v[32];
                ptx::tmem_ld32(tmem + lane_off + 32 * cb, v);
                ptx::tmem_ld_wait();
                uint32_t ph[16], pl[16];
#pragma unroll
                for (int jj = 0; jj < 32; jj += 2) {
                    const int j = 32 * cb + jj;
                    float e0 = 0.f, e1 = 0.f;
                    // the causal selection before the exponent
                    if (!diag || j <= i)
                        e0 = __uint_as_float(v[jj]) * exp2f(g_i - gj[s * 128 + j]) * dtj[s * 128 + j];
                    if (!diag || j + 1 <= i)
                        e1 = __uint_as_float(v[jj + 1]) * exp2f(g_i - gj[s * 128 + j + 1]) *
                             dtj[s * 128 + j + 1];
                    split2(e0, e1, ph[jj >> 1], pl[jj >> 1]);
                }
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int ch = 4 * cb + q;   // 16-byte chunk 0..15 of the row
                    const int kb = ch >> 3, c8 = ch & 7;
                    const int off = kb * 16384 + ((c8 ^ (i & 7)) << 4);
                    *reinterpret_cast<uint4 *>(Lh + off) =
                        make_uint4(ph[4 * q], ph[4 * q + 1], ph[4 * q + 2], ph[4 * q + 3]);
                    *reinterpret_cast<uint4 *>(Ll + off) =
                        make_uint4(pl[4 * q], pl[4 * q + 1], pl[4 * q + 2], pl[4 * q + 3]);
                }
            }
            ptx::fence_proxy_async_smem();
            ptx::tc_fence_before();
            ptx::mbar_arrive(bar_L);
        }
        const bool go = __all_sync(0xffffffffu, ok && ptx::mbar_wait(bar_acc, 0));
        if (go) {
            ptx::tc_fence_after();
            const int64_t t = c * Q + r * 128 + i;
            const float e_i = exp2f(g_i);
            const float Dh = p.D && SSD_IDX_OK(p.err, h, p.H) ? p.D[h] : 0.f;
            const uint8_t *Xh = smem + SM::kX + i * 128;
            const uint8_t *Xl = Xh + 16384;
            const int64_t yo = b * p.y_sb + t * p.y_sl + int64_t(h) * p.y_sh;
            float *yrow = p.y + yo;
#pragma unroll 1
            for (int cb = 0; cb < 2; ++cb) {
                uint32_t a[32], d[32];
                ptx::tmem_ld32(t_inter + lane_off + 32 * cb, a);
                ptx::tmem_ld32(t_intra + lane_off + 32 * cb, d);
                ptx::tmem_ld_wait();
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int ch = 4 * cb + q;   // 8 headdim values per 16-byte chunk
                    const int off = (ch ^ (i & 7)) << 4;
                    const uint4 xh = *reinterpret_cast<const uint4 *>(Xh + off);
                    const uint4 xl = *reinterpret_cast<const uint4 *>(Xl + off);
                    const uint32_t *uh = reinterpret_cast<const uint32_t *>(&xh);
                    const uint32_t *ul = reinterpret_cast<const uint32_t *>(&xl);
                    float o[8];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const float2 xf = join2(uh[k], ul[k]);
                        const int jj = 8 * q + 2 * k;
                        o[2 * k] = fmaf(e_i, __uint_as_float(a[jj]), __uint_as_float(d[jj])) + Dh * xf.x;
                        o[2 * k + 1] =
                            fmaf(e_i, __uint_as_float(a[jj + 1]), __uint_as_float(d[jj + 1])) + Dh * xf.y;
                    }
                    if (t < p.L && SSD_IDX_OK(p.err, yo + 8 * ch + 7, p.n_y)) {
                        *reinterpret_cast<float4 *>(yrow + 8 * ch) = make_float4(o[0], o[1], o[2], o[3]);
                        *reinterpret_cast<float4 *>(yrow + 8 * ch + 4) = make_float4(o[4], o[5], o[6], o[7]);
                    }
                }
            }
        } else {
            ok = false;
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

cudaError_t split(const float *src, int64_t n0, int64_t n1, int64_t n2, int64_t inner, int64_t s0,
                  int64_t s1, int64_t s2, __nv_bfloat16 *hi, __nv_bfloat16 *lo, unsigned int *err,
                  cudaStream_t st) {
    const int64_t total = n0 * n1 * n2 * inner;
    if (total <= 0) return cudaSuccess;
    const int64_t n_src = (n0 - 1) * s0 + (n1 - 1) * s1 + (n2 - 1) * s2 + inner;
    const int64_t blocks = (total + 255) / 256;
    const unsigned grid = unsigned(blocks < 152 * 16 ? blocks : 152 * 16);
    k_split_hilo<<<grid, 256, 0, st>>>(src, n1, n2, inner, s0, s1, s2, total, hi, lo, err, n_src);
    return cudaGetLastError();
}

// Contiguous bf16 [n3][n2][n1][inner] tensor map with box {64, 1, rows, 1}.
cudaError_t tmap_contig_4d(CUtensorMap *m, const void *base, int64_t n3, int64_t n2, int64_t n1,
                           int64_t inner, uint32_t rows) {
    const uint64_t dims[4] = {uint64_t(inner), uint64_t(n1), uint64_t(n2), uint64_t(n3)};
    const uint64_t strides[3] = {uint64_t(inner) * 2, uint64_t(n1 * inner) * 2,
                                 uint64_t(n2 * n1 * inner) * 2};
    const uint32_t box[4] = {64, 1, rows, 1};
    return make_tmap_bf16(m, base, 4, dims, strides, box);
}

}  // namespace

bool tc_f32_supported(const Dims &d, int xdt) {
    return xdt == DT_F32 && d.P == 64 && d.N == 128 && (d.Q == 128 || d.Q == 256) && d.L > 0;
}

cudaError_t split_inputs_f32(const Args &a, cudaStream_t s) {
    const Dims &d = a.d;
    unsigned int *err = nullptr;
    cudaError_t e = device_error_word(&err);
    if (e != cudaSuccess) return e;
    auto *xh = static_cast<__nv_bfloat16 *>(a.f32s.x_hi), *xl = static_cast<__nv_bfloat16 *>(a.f32s.x_lo);
    auto *bh = static_cast<__nv_bfloat16 *>(a.f32s.b_hi), *bl = static_cast<__nv_bfloat16 *>(a.f32s.b_lo);
    auto *ch = static_cast<__nv_bfloat16 *>(a.f32s.c_hi), *cl = static_cast<__nv_bfloat16 *>(a.f32s.c_lo);
    if ((e = split(static_cast<const float *>(a.x), d.B, d.L, d.H, d.P, a.x_sb, a.x_sl, a.x_sh, xh, xl,
                   err, s)))
        return e;
    if ((e = split(static_cast<const float *>(a.Bm), d.B, d.L, d.G, d.N, a.b_sb, a.b_sl, a.b_sg, bh,
                   bl, err, s)))
        return e;
    return split(static_cast<const float *>(a.Cm), d.B, d.L, d.G, d.N, a.c_sb, a.c_sl, a.c_sg, ch, cl,
                 err, s);
}

cudaError_t tc_chunk_state_f32(const Args &a, cudaStream_t s) {
    const Dims &d = a.d;
    CUtensorMap tm_xh, tm_xl, tm_bh, tm_bl;
    cudaError_t e;
    if ((e = tmap_contig_4d(&tm_xh, a.f32s.x_hi, d.B, d.L, d.H, 64, 64))) return e;
    if ((e = tmap_contig_4d(&tm_xl, a.f32s.x_lo, d.B, d.L, d.H, 64, 64))) return e;
    if ((e = tmap_contig_4d(&tm_bh, a.f32s.b_hi, d.B, d.L, d.G, 128, 64))) return e;
    if ((e = tmap_contig_4d(&tm_bl, a.f32s.b_lo, d.B, d.L, d.G, 128, 64))) return e;
    unsigned int *err = nullptr;
    if ((e = device_error_word(&err)) != cudaSuccess) return e;
    Args ax = a;
    fill_extents(ax);
    StateF32Params p{d.L, d.Lp(), int(d.H), int(d.hpg()), int(d.Q), a.dt, a.dt_sb, a.dt_sl,
                     a.G, a.S, d.nc, err, ax.n_dt, d.B * d.H * d.Lp(),
                     d.B * d.nc * d.H * 64 * 128};
    if (d.hpg() % 2 == 0) {
        auto k = k_chunk_state_tc_f32<2, 2>;
        const int smem = StateF32Smem<2, 2>::kBytes;
        if ((e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem))) return e;
        k<<<dim3(unsigned(d.nc), unsigned(d.H / 2), unsigned(d.B)), 192, smem, s>>>(tm_xh, tm_xl,
                                                                                    tm_bh, tm_bl, p);
    } else {
        auto k = k_chunk_state_tc_f32<1, 2>;
        const int smem = StateF32Smem<1, 2>::kBytes;
        if ((e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem))) return e;
        k<<<dim3(unsigned(d.nc), unsigned(d.H), unsigned(d.B)), 192, smem, s>>>(tm_xh, tm_xl, tm_bh,
                                                                                tm_bl, p);
    }
    return cudaGetLastError();
}

cudaError_t tc_chunk_scan_f32(const Args &a, cudaStream_t s) {
    const Dims &d = a.d;
    unsigned int *err = nullptr;
    cudaError_t e = device_error_word(&err);
    if (e != cudaSuccess) return e;
    // h_prev (fp32, contiguous [B, nc, H, P, N]) -> hi, lo
    auto *hh = static_cast<__nv_bfloat16 *>(a.f32s.hp_hi), *hl = static_cast<__nv_bfloat16 *>(a.f32s.hp_lo);
    if ((e = split(static_cast<const float *>(a.h_prev), d.B * d.nc, d.H, d.P, d.N, d.H * d.P * d.N,
                   d.P * d.N, d.N, hh, hl, err, s)))
        return e;
    CUtensorMap tm_xh, tm_xl, tm_bh, tm_bl, tm_ch, tm_cl, tm_hh, tm_hl;
    if ((e = tmap_contig_4d(&tm_xh, a.f32s.x_hi, d.B, d.L, d.H, 64, 128))) return e;
    if ((e = tmap_contig_4d(&tm_xl, a.f32s.x_lo, d.B, d.L, d.H, 64, 128))) return e;
    if ((e = tmap_contig_4d(&tm_bh, a.f32s.b_hi, d.B, d.L, d.G, 128, 128))) return e;
    if ((e = tmap_contig_4d(&tm_bl, a.f32s.b_lo, d.B, d.L, d.G, 128, 128))) return e;
    if ((e = tmap_contig_4d(&tm_ch, a.f32s.c_hi, d.B, d.L, d.G, 128, 128))) return e;
    if ((e = tmap_contig_4d(&tm_cl, a.f32s.c_lo, d.B, d.L, d.G, 128, 128))) return e;
    // h_prev hi / lo [B, nc, H, P, N] viewed as rows of N: {N, B*nc*H*P, 1}
    const uint64_t hd[3] = {128, uint64_t(d.B * d.nc * d.H * 64), 1};
    const uint64_t hs[2] = {128 * 2, uint64_t(d.B * d.nc * d.H * 64) * 256};
    const uint32_t hbox[3] = {64, 64, 1};
    if ((e = make_tmap_bf16(&tm_hh, hh, 3, hd, hs, hbox))) return e;
    if ((e = make_tmap_bf16(&tm_hl, hl, 3, hd, hs, hbox))) return e;
    Args ax = a;
    fill_extents(ax);
    ScanF32Params p{d.L, d.Lp(), d.nc, int(d.H), int(d.hpg()), int(d.Q), a.dt, a.dt_sb, a.dt_sl,
                    a.G, a.D, static_cast<float *>(a.y), a.y_sb, a.y_sl, a.y_sh, err, ax.n_dt,
                    d.B * d.H * d.Lp(), ax.n_y};
    const int smem = ScanF32Smem::kBytes;
    if ((e = cudaFuncSetAttribute(k_chunk_scan_tc_f32, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  smem)))
        return e;
    k_chunk_scan_tc_f32<<<dim3(unsigned(d.nc * (d.Q / 128)), unsigned(d.H), unsigned(d.B)), 192, smem,
                          s>>>(tm_xh, tm_xl, tm_bh, tm_bl, tm_ch, tm_cl, tm_hh, tm_hl, p);
    return cudaGetLastError();
}

}  // namespace ssd
