// Decode steps of the Mamba-2 layer -- the selective state update of
// "Optimizing Nemotron v3 Super in TensorRT-LLM", section 6.1 "The SSU Math",
// with the dt bias, softplus and z gate of section 6.2's reference, applied
// to T tokens per sequence in one launch as in section 10.4 "Multi-Token
// State Update Kernel":
//     dt' = softplus(dt + dt_bias)          (each step optional)
//     state = exp(A dt') state + dt' x (outer) B
//     out   = (state C + D x) * silu(z)
// for every (batch, head), head h reading group h / (H / G); token t > 0 may
// start from the cached state after an earlier token (its parent) instead of
// the one after token t - 1.  With slot indices (the serving kernel's
// state_batch_idx of section 10.4) sequence b's state and cache live in slot
// slots[b] of a pool; a row whose slot is outside the pool is padding and is
// skipped.
//
// The state is kept in fp32 or, as in section 6.4.3's Blackwell path for
// 16-bit state caches, in bf16: each token's update is computed in fp32 from
// the kept values, its output from the unrounded result, and what is kept (the
// tile, the per-token cache, the final state) is rounded to nearest even.
//
// The step reads and writes the state once per call, whatever T, and
// everything else is a few hundred bytes per head and token, so it is bound
// by HBM.  Each CTA owns a tile of state rows of one (batch, head): one
// elected thread brings the whole tile into shared memory with bulk copies,
// the T tokens update it there in place (each thread four consecutive
// columns of its rows), and one bulk copy writes it back, so neither
// direction holds registers and an SM keeps six tiles in flight.  The
// per-token state cache is written with coalesced 16-byte stores.  A row's
// output is a shuffle reduction over the lanes holding it.  No tensor cores:
// the only contraction is a length-N dot product per row.
#include "ptx_sm100.cuh"
#include "ssd_decode.h"

#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace ssd {
namespace {

constexpr int kSsuThreads = 128;
constexpr int kMaxRT = 16;                 // passes of rows per tile at most (32 KB at N = 128)
constexpr uint32_t kBulkChunk = 16384;     // bytes per bulk copy
constexpr unsigned kErrTimeout = 1u;       // same bit as the fused forward's

// Shared -> global bulk copy of `bytes` (16-byte aligned addresses, a multiple
// of 16 bytes), tracked by this thread's bulk-async group.
__device__ __forceinline__ void bulk_store(void *dst, const void *src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst),
                 "r"(ptx::smem_u32(src)), "r"(bytes)
                 : "memory");
}

template <typename T>
__device__ __forceinline__ float to_f(T v);
template <>
__device__ __forceinline__ float to_f<float>(float v) { return v; }
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T>
__device__ __forceinline__ T from_f(float v);
template <>
__device__ __forceinline__ float from_f<float>(float v) { return v; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float v) {
    return __float2bfloat16_rn(v);
}

// Four consecutive state elements as stored (16 bytes for f32, 8 for bf16)
// and as computed on.
template <typename S>
struct State4;
template <>
struct State4<float> {
    using V = float4;
    static __device__ __forceinline__ float4 get(V v) { return v; }
    static __device__ __forceinline__ V put(float4 v) { return v; }
};
template <>
struct State4<__nv_bfloat16> {
    using V = uint2;
    static __device__ __forceinline__ float4 get(V v) {
        const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&v.x));
        const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&v.y));
        return make_float4(lo.x, lo.y, hi.x, hi.y);
    }
    static __device__ __forceinline__ V put(float4 v) {
        const __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y);
        const __nv_bfloat162 hi = __floats2bfloat162_rn(v.z, v.w);
        return make_uint2(*reinterpret_cast<const uint32_t *>(&lo),
                          *reinterpret_cast<const uint32_t *>(&hi));
    }
};

// four consecutive elements of a B / C row (16-byte aligned for f32, 8 for bf16)
__device__ __forceinline__ float4 load4(const float *p) {
    return *reinterpret_cast<const float4 *>(p);
}
__device__ __forceinline__ float4 load4(const __nv_bfloat16 *p) {
    const uint2 u = *reinterpret_cast<const uint2 *>(p);
    const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.x));
    const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.y));
    return make_float4(lo.x, lo.y, hi.x, hi.y);
}

// grid (P / R, H, B), block kSsuThreads = kRowsPass x (N / 4) threads,
// dynamic shared memory R N sizeof(S) bytes.  R = rows: a multiple of kRowsPass of at
// most kMaxRT kRowsPass, or all P rows when P < kRowsPass.  Thread (rr, c)
// owns columns 4c .. 4c + 3 of the local rows rr + i kRowsPass below R.
// Each token's x and gate silu(z) of the tile's rows are staged in shared
// memory, and each row's sum over n is left there for the threads that write
// the outputs out coalesced a token later (all three double-buffered by token
// parity): the pass loop itself holds no per-row epilogue.
template <int N, typename T, typename S>
__global__ void __launch_bounds__(kSsuThreads)
k_ssu_tokens(const SsuArgs a, int rows, unsigned int *err) {
    constexpr int kTpr = N / 4;                     // threads per state row
    constexpr int kRowsPass = kSsuThreads / kTpr;   // rows per pass
    using SV = State4<S>;
    using V = typename SV::V;
    extern __shared__ __align__(16) float4 smem_tile[];
    V *tile = reinterpret_cast<V *>(smem_tile);
    __shared__ uint64_t full;
    __shared__ float xs[2][128], gs[2][128], ps[2][128];   // rows <= P <= 128
    const int b = blockIdx.z, h = blockIdx.y;
    int64_t slot = b;                               // where row b's state and cache live
    if (a.slots) {
        slot = a.slots[b];
        if (slot < 0 || slot >= a.S) return;        // a padding row: nothing read or written
    }
    const int g = h / (a.H / a.G);
    const int r0 = blockIdx.x * rows;
    const int c = threadIdx.x % kTpr, rr = threadIdx.x / kTpr;
    const int nrt = (rows + kRowsPass - 1) / kRowsPass;   // uniform over the CTA
    const size_t head = size_t(slot) * a.H + h;
    S *st = static_cast<S *>(a.state) + (head * a.P + r0) * N;
    const uint32_t bytes = uint32_t(rows) * N * uint32_t(sizeof(S));

    if (threadIdx.x == 0) {
        ptx::mbar_init(&full, 1);
        ptx::fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        ptx::mbar_arrive_expect_tx(&full, bytes);
        for (uint32_t off = 0; off < bytes; off += kBulkChunk)
            ptx::bulk_load(reinterpret_cast<char *>(tile) + off,
                           reinterpret_cast<const char *>(st) + off,
                           bytes - off < kBulkChunk ? bytes - off : kBulkChunk, &full);
    }
    const float Ah = a.A[h];
    const float Dh = a.D ? a.D[h] : 0.f;
    const float bias = a.dt_bias ? a.dt_bias[h] : 0.f;
    // token t's x and silu(z) (1 without z) of this tile's rows into buffer t & 1;
    // thread r stages row r and, a token later, writes its output
    auto stage_xz = [&](int t) {
        if (threadIdx.x < rows) {
            const int row = r0 + threadIdx.x;
            xs[t & 1][threadIdx.x] = to_f(static_cast<const T *>(a.x)[
                int64_t(b) * a.x_sb + int64_t(t) * a.x_st + int64_t(h) * a.x_sh + row]);
            float gate = 1.f;
            if (a.z) {
                const float zv = to_f(static_cast<const T *>(a.z)[
                    int64_t(b) * a.z_sb + int64_t(t) * a.z_st + int64_t(h) * a.z_sh + row]);
                gate = zv / (1.f + expf(-zv));
            }
            gs[t & 1][threadIdx.x] = gate;
        }
    };
    // token t's outputs from buffer t & 1: (sum_n + D x) silu(z)
    auto write_out = [&](int t) {
        if (threadIdx.x < rows) {
            const int i = threadIdx.x;
            const float o = fmaf(Dh, xs[t & 1][i], ps[t & 1][i]) * gs[t & 1][i];
            static_cast<T *>(a.out)[int64_t(b) * a.o_sb + int64_t(t) * a.o_st +
                                    int64_t(h) * a.o_sh + r0 + i] = from_f<T>(o);
        }
    };
    // token t's dt, and this thread's four columns of its B and C rows
    const float *dtp = a.dt + int64_t(b) * a.dt_sb + h;
    const T *bp = static_cast<const T *>(a.Bm) + int64_t(b) * a.bc_sb + int64_t(g) * a.bc_sg + 4 * c;
    const T *cp = static_cast<const T *>(a.Cm) + int64_t(b) * a.bc_sb + int64_t(g) * a.bc_sg + 4 * c;
    // token 0's inputs are in flight with the state copy; each token fetches the next one's
    stage_xz(0);
    float dn = dtp[0];
    float4 bn = load4(bp), cn = load4(cp);
    if (!ptx::mbar_wait(&full, 0)) {   // uniform: every thread gives up on the same copy
        if (threadIdx.x == 0) atomicOr(err, kErrTimeout);
        return;
    }
    for (int t = 0; t < a.T; ++t) {
        float d = dn + bias;
        const float4 bq = bn, cq = cn;
        if (t + 1 < a.T) {
            dn = dtp[int64_t(t + 1) * a.dt_st];
            bn = load4(bp + int64_t(t + 1) * a.bc_st);
            cn = load4(cp + int64_t(t + 1) * a.bc_st);
        }
        if (a.parent && t > 0) {
            // start from the state after the parent token, when it is an earlier one
            // (each thread reloads its own entries of the tile)
            const int pt = a.parent[int64_t(b) * a.par_sb + t];
            if (pt >= 0 && pt < t) {
                const S *src = static_cast<const S *>(a.inter) +
                               ((slot * a.T + pt) * a.H + h) * a.P * N;
                for (int i = 0; i < nrt; ++i) {
                    const int lr = rr + i * kRowsPass;
                    if (lr < rows)
                        tile[lr * kTpr + c] = *reinterpret_cast<const V *>(
                            src + int64_t(r0 + lr) * N + 4 * c);
                }
            }
        }
        if (a.softplus) d = d <= 20.f ? log1pf(expf(d)) : d;   // log(1 + e^d), = d to fp32 above 20
        const float dA = expf(Ah * d);
        __syncthreads();                            // token t staged, token t - 1 summed
        if (t > 0) write_out(t - 1);
        if (t + 1 < a.T) stage_xz(t + 1);           // the other buffer, read after the next sync
        const float *xt = xs[t & 1];
        float *sums = ps[t & 1];
        S *ir = a.inter ? static_cast<S *>(a.inter) + ((slot * a.T + t) * a.H + h) * a.P * N
                        : nullptr;
#pragma unroll 4
        for (int i = 0; i < nrt; ++i) {
            const int lr = rr + i * kRowsPass;        // local row
            const bool live = lr < rows;              // false only when P < kRowsPass
            float partial = 0.f;
            if (live) {
                const float u = d * xt[lr];
                float4 v = SV::get(tile[lr * kTpr + c]);
                v.x = fmaf(v.x, dA, u * bq.x);
                v.y = fmaf(v.y, dA, u * bq.y);
                v.z = fmaf(v.z, dA, u * bq.z);
                v.w = fmaf(v.w, dA, u * bq.w);
                const V kept = SV::put(v);          // the output below uses v unrounded
                tile[lr * kTpr + c] = kept;
                if (ir) *reinterpret_cast<V *>(ir + int64_t(r0 + lr) * N + 4 * c) = kept;
                partial = fmaf(v.x, cq.x, fmaf(v.y, cq.y, fmaf(v.z, cq.z, v.w * cq.w)));
            }
            // sum over the row's kTpr lanes (contiguous within the warp)
#pragma unroll
            for (int off = kTpr / 2; off > 0; off >>= 1)
                partial += __shfl_xor_sync(0xffffffffu, partial, off);
            if (live && c == 0) sums[lr] = partial;
        }
    }
    // every thread's tile writes, then one bulk copy back (its shared-memory
    // reads must finish before the CTA leaves); the last token's outputs
    if (a.update) ptx::fence_proxy_async_smem();
    __syncthreads();
    write_out(a.T - 1);
    if (a.update) {
        if (threadIdx.x == 0) {
            for (uint32_t off = 0; off < bytes; off += kBulkChunk)
                bulk_store(reinterpret_cast<char *>(st) + off, reinterpret_cast<char *>(tile) + off,
                           bytes - off < kBulkChunk ? bytes - off : kBulkChunk);
            ptx::bulk_commit_group();
            ptx::bulk_wait_group_read0();
        }
    }
}

int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
        cudaGetLastError();
        return 152;
    }
    return n;
}

template <int N, typename T, typename S>
cudaError_t launch_n(const SsuArgs &a, cudaStream_t s) {
    constexpr int kRowsPass = kSsuThreads / (N / 4);
    // tiles of at most kMaxRT passes of rows (32 KB of fp32 at N = 128), halved while the grid is
    // below two CTAs per SM (few sequences: spread the rows over more SMs)
    int rows = a.P < kMaxRT * kRowsPass ? a.P : kMaxRT * kRowsPass;   // P / rows whole
    const int64_t want = 2 * int64_t(sm_count());
    while (rows / 2 >= kRowsPass && int64_t(a.B) * a.H * (a.P / rows) < want) rows /= 2;
    unsigned int *err = nullptr;
    cudaError_t e = device_error_word(&err);
    if (e != cudaSuccess) return e;
    const dim3 grid(unsigned(a.P / rows), unsigned(a.H), unsigned(a.B));
    k_ssu_tokens<N, T, S><<<grid, kSsuThreads, size_t(rows) * N * sizeof(S), s>>>(a, rows, err);
    return cudaGetLastError();
}

template <typename T, typename S>
cudaError_t launch_t(const SsuArgs &a, cudaStream_t s) {
    switch (a.N) {
    case 16: return launch_n<16, T, S>(a, s);
    case 32: return launch_n<32, T, S>(a, s);
    case 64: return launch_n<64, T, S>(a, s);
    case 128: return launch_n<128, T, S>(a, s);
    default: return cudaErrorInvalidValue;
    }
}

template <typename T>
cudaError_t launch_s(const SsuArgs &a, cudaStream_t s) {
    return a.sdt == DT_BF16 ? launch_t<T, __nv_bfloat16>(a, s) : launch_t<T, float>(a, s);
}

}  // namespace

cudaError_t launch_ssu(const SsuArgs &a, cudaStream_t s) {
    if (a.B == 0 || a.T == 0) return cudaSuccess;
    return a.xdt == DT_BF16 ? launch_s<__nv_bfloat16>(a, s) : launch_s<float>(a, s);
}

}  // namespace ssd
