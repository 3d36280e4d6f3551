// Host side of the C ABI declared in include/ssd.h: argument checks, the
// workspace plan and the ordered launch of the four steps on the caller's
// stream.  Every check runs before the first launch; nothing here allocates,
// frees or synchronises.
#include "ssd.h"
#include "ssd_decode.h"
#include "ssd_internal.h"
#include "ssd_mixer.h"
#include "ssd_tc.cuh"

#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <initializer_list>
#include <string>

namespace {

thread_local std::string g_detail;

ssd_status fail(ssd_status st, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_detail = buf;
    return st;
}

ssd_status ok() {
    g_detail.clear();
    return SSD_OK;
}

size_t elem_size(int dt) { return dt == SSD_BF16 ? 2 : 4; }
size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

bool supported_dim(int64_t v) { return v == 16 || v == 32 || v == 64 || v == 128; }
bool supported_chunk(int64_t q) { return q == 64 || q == 128 || q == 256; }

// Address range [lo, hi) a tensor touches; empty when any extent is 0.
struct Range {
    uintptr_t lo = 0, hi = 0;
};
Range range_of(const ssd_tensor *t) {
    Range r;
    if (!t || !t->data) return r;
    int64_t last = 0;
    for (int i = 0; i < t->ndim; ++i) {
        if (t->shape[i] == 0) return r;
        last += (t->shape[i] - 1) * t->stride[i];
    }
    r.lo = reinterpret_cast<uintptr_t>(t->data);
    r.hi = r.lo + size_t(last + 1) * elem_size(t->dtype);
    return r;
}
Range range_raw(const void *p, size_t bytes) {
    Range r;
    if (p && bytes) {
        r.lo = reinterpret_cast<uintptr_t>(p);
        r.hi = r.lo + bytes;
    }
    return r;
}
bool overlap(Range a, Range b) {
    return a.lo < a.hi && b.lo < b.hi && a.lo < b.hi && b.lo < a.hi;
}

// Checks one tensor's rank, dtype, shape, unit inner stride and alignment.
// dtype < 0 accepts f32 or bf16 (int32 only where asked for by name).
// contiguous demands packed row-major strides.
ssd_status check_tensor(const ssd_tensor *t, const char *name, int ndim,
                        const int64_t *shape, int dtype, bool contiguous,
                        bool align_strides16) {
    if (!t) return fail(SSD_ERR_INVALID_ARG, "%s: null tensor descriptor", name);
    if (t->ndim != ndim)
        return fail(SSD_ERR_INVALID_ARG, "%s: ndim %d, expected %d", name, t->ndim, ndim);
    auto dname = [](int d) { return d == SSD_F32 ? "f32" : d == SSD_BF16 ? "bf16" : "i32"; };
    if (t->dtype != SSD_F32 && t->dtype != SSD_BF16 && t->dtype != SSD_I32)
        return fail(SSD_ERR_INVALID_ARG, "%s: unknown dtype code %d", name, t->dtype);
    if ((dtype >= 0 && t->dtype != dtype) || (dtype < 0 && t->dtype == SSD_I32))
        return fail(SSD_ERR_INVALID_ARG, "%s: dtype %s, expected %s", name, dname(t->dtype),
                    dtype >= 0 ? dname(dtype) : "f32 or bf16");
    int64_t numel = 1;
    for (int i = 0; i < ndim; ++i) {
        if (t->shape[i] != shape[i])
            return fail(SSD_ERR_INVALID_ARG, "%s: shape[%d] = %lld, expected %lld", name, i,
                        (long long)t->shape[i], (long long)shape[i]);
        numel *= shape[i];
    }
    if (numel > 0 && !t->data) return fail(SSD_ERR_INVALID_ARG, "%s: null data pointer", name);
    if (t->stride[ndim - 1] != 1 && shape[ndim - 1] > 1)
        return fail(SSD_ERR_INVALID_ARG, "%s: innermost stride %lld, must be 1", name,
                    (long long)t->stride[ndim - 1]);
    if (contiguous) {
        int64_t want = 1;
        for (int i = ndim - 1; i >= 0; --i) {
            if (shape[i] > 1 && t->stride[i] != want)
                return fail(SSD_ERR_INVALID_ARG, "%s: must be contiguous (stride[%d] = %lld, "
                            "expected %lld)", name, i, (long long)t->stride[i], (long long)want);
            want *= shape[i];
        }
    }
    for (int i = 0; i < ndim - 1; ++i)
        if (t->stride[i] < 0)
            return fail(SSD_ERR_INVALID_ARG, "%s: negative stride", name);
    const size_t es = elem_size(t->dtype);
    if (numel > 0 && (reinterpret_cast<uintptr_t>(t->data) % (align_strides16 ? 16 : es)))
        return fail(SSD_ERR_ALIGNMENT, "%s: base pointer %p not %zu-byte aligned", name, t->data,
                    align_strides16 ? size_t(16) : es);
    if (align_strides16)
        for (int i = 0; i < ndim - 1; ++i)
            if (shape[i] > 1 && (t->stride[i] * int64_t(es)) % 16)
                return fail(SSD_ERR_ALIGNMENT, "%s: stride[%d] = %lld elements is not a multiple "
                            "of 16 bytes", name, i, (long long)t->stride[i]);
    return SSD_OK;
}

ssd_status check_geometry(int64_t B, int64_t L, int64_t H, int64_t P, int64_t N, int64_t G,
                          int64_t Q) {
    if (B < 0 || L < 0) return fail(SSD_ERR_INVALID_ARG, "batch %lld / seqlen %lld negative",
                                    (long long)B, (long long)L);
    if (H <= 0 || G <= 0) return fail(SSD_ERR_INVALID_ARG, "nheads %lld / ngroups %lld must be "
                                      "positive", (long long)H, (long long)G);
    if (H % G) return fail(SSD_ERR_INVALID_ARG, "nheads %lld is not a multiple of ngroups %lld",
                           (long long)H, (long long)G);
    if (Q <= 0) return fail(SSD_ERR_INVALID_ARG, "chunk_size %lld must be positive", (long long)Q);
    if (!supported_chunk(Q))
        return fail(SSD_ERR_UNSUPPORTED, "chunk_size %lld unsupported (64, 128 or 256)",
                    (long long)Q);
    if (!supported_dim(P))
        return fail(SSD_ERR_UNSUPPORTED, "headdim %lld unsupported (16, 32, 64 or 128)",
                    (long long)P);
    if (!supported_dim(N))
        return fail(SSD_ERR_UNSUPPORTED, "dstate %lld unsupported (16, 32, 64 or 128)",
                    (long long)N);
    if (B > 65535 || H > 65535)
        return fail(SSD_ERR_UNSUPPORTED, "batch %lld or nheads %lld above 65535", (long long)B,
                    (long long)H);
    const int64_t nc = (L + Q - 1) / Q;
    if (nc > (int64_t(1) << 30))
        return fail(SSD_ERR_UNSUPPORTED, "seqlen %lld too long", (long long)L);
    return SSD_OK;
}

// Either the fused path (workspace only for a split last wave) or the
// four-step path with its intermediates in the workspace.
struct Plan {
    bool fused;
    bool f32_split;   // fp32 on the tensor cores: bf16 hi / lo copies follow h_prev
    size_t off_G, off_S, off_hp, total;
    size_t off_x_hi, off_x_lo, off_b_hi, off_b_lo, off_c_hi, off_c_lo, off_hp_hi, off_hp_lo;
};

Plan plan_workspace(const ssd::Dims &d, int xdt) {
    Plan p{};
    p.fused = ssd::use_fused(d, xdt);
    if (p.fused) {
        // only a split last wave needs scratch (the tail segments' states)
        p.total = (ssd::pair_supported(d, xdt) ? ssd::pair_split(d, ssd::device_sm_count())
                                               : ssd::fused_split(d, ssd::device_sm_count()))
                      .ws_bytes;
        return p;
    }
    const size_t g = size_t(d.B) * d.H * d.nc * d.Q * 4;
    const size_t s = size_t(d.B) * d.nc * d.H * d.P * d.N * 4;
    const size_t hp = size_t(d.B) * d.nc * d.H * d.P * d.N * elem_size(xdt);
    p.off_G = 0;
    p.off_S = align256(p.off_G + g);
    p.off_hp = align256(p.off_S + s);
    p.total = align256(p.off_hp + hp);
    p.f32_split = ssd::f32_split_plan(d, xdt);
    if (p.f32_split) {
        const size_t xb = size_t(d.B) * d.L * d.H * d.P * 2, bb = size_t(d.B) * d.L * d.G * d.N * 2,
                     hb = size_t(d.B) * d.nc * d.H * d.P * d.N * 2;
        p.off_x_hi = p.total;
        p.off_x_lo = align256(p.off_x_hi + xb);
        p.off_b_hi = align256(p.off_x_lo + xb);
        p.off_b_lo = align256(p.off_b_hi + bb);
        p.off_c_hi = align256(p.off_b_lo + bb);
        p.off_c_lo = align256(p.off_c_hi + bb);
        p.off_hp_hi = align256(p.off_c_lo + bb);
        p.off_hp_lo = align256(p.off_hp_hi + hb);
        p.total = align256(p.off_hp_lo + hb);
    }
    return p;
}

// Every data pointer must be device (or managed) memory of the current
// device: a host pointer handed to a kernel would fault it.  Runs after all
// pure-host checks, so argument errors are reported without touching CUDA.
struct NamedPtr {
    const void *p;
    const char *name;
};
ssd_status check_device_ptrs(std::initializer_list<NamedPtr> ptrs) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(SSD_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    for (const NamedPtr &np : ptrs) {
        if (!np.p) continue;
        cudaPointerAttributes at{};
        e = cudaPointerGetAttributes(&at, np.p);
        if (e != cudaSuccess) {
            cudaGetLastError();
            return fail(SSD_ERR_INVALID_ARG, "%s: pointer %p is not CUDA memory (%s)", np.name,
                        np.p, cudaGetErrorString(e));
        }
        if (at.type == cudaMemoryTypeManaged) continue;
        if (at.type != cudaMemoryTypeDevice)
            return fail(SSD_ERR_INVALID_ARG, "%s: pointer %p is host memory; device memory is "
                        "required", np.name, np.p);
        if (at.device != dev)
            return fail(SSD_ERR_INVALID_ARG, "%s: pointer on device %d, current device is %d",
                        np.name, at.device, dev);
    }
    return SSD_OK;
}

ssd_status cuda_status(cudaError_t e, const char *what) {
    if (e == cudaSuccess) return SSD_OK;
    return fail(SSD_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

void fill_x(ssd::Args &a, const ssd_tensor *x) {
    a.x = x->data;
    a.x_sb = x->stride[0];
    a.x_sl = x->stride[1];
    a.x_sh = x->stride[2];
}
void fill_dt(ssd::Args &a, const ssd_tensor *dt) {
    a.dt = static_cast<const float *>(dt->data);
    a.dt_sb = dt->stride[0];
    a.dt_sl = dt->stride[1];
}
void fill_bc(ssd::Args &a, const ssd_tensor *Bm, const ssd_tensor *Cm) {
    if (Bm) {
        a.Bm = Bm->data;
        a.b_sb = Bm->stride[0];
        a.b_sl = Bm->stride[1];
        a.b_sg = Bm->stride[2];
    }
    if (Cm) {
        a.Cm = Cm->data;
        a.c_sb = Cm->stride[0];
        a.c_sl = Cm->stride[1];
        a.c_sg = Cm->stride[2];
    }
}
void fill_y(ssd::Args &a, ssd_tensor *y) {
    a.y = y->data;
    a.y_sb = y->stride[0];
    a.y_sl = y->stride[1];
    a.y_sh = y->stride[2];
}

}  // namespace

namespace ssd {
void set_error_detail(const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_detail = buf;
}
}  // namespace ssd

extern "C" {

const char *ssd_status_string(ssd_status s) {
    switch (s) {
        case SSD_OK: return "SSD_OK";
        case SSD_ERR_INVALID_ARG: return "SSD_ERR_INVALID_ARG";
        case SSD_ERR_UNSUPPORTED: return "SSD_ERR_UNSUPPORTED";
        case SSD_ERR_ALIGNMENT: return "SSD_ERR_ALIGNMENT";
        case SSD_ERR_WORKSPACE: return "SSD_ERR_WORKSPACE";
        case SSD_ERR_CUDA: return "SSD_ERR_CUDA";
        case SSD_ERR_TIMEOUT: return "SSD_ERR_TIMEOUT";
        case SSD_ERR_DEVICE_BOUNDS: return "SSD_ERR_DEVICE_BOUNDS";
    }
    return "SSD_UNKNOWN_STATUS";
}

const char *ssd_last_error_detail(void) { return g_detail.c_str(); }

const char *ssd_describe_plan(int64_t batch, int64_t seqlen, int64_t nheads, int64_t headdim,
                              int64_t dstate, int64_t ngroups, int64_t chunk_size,
                              int32_t x_dtype) {
    thread_local std::string text;
    if (x_dtype != SSD_F32 && x_dtype != SSD_BF16) {
        text = "rejected: unknown dtype code";
        return text.c_str();
    }
    const std::string saved = g_detail;
    if (check_geometry(batch, seqlen, nheads, headdim, dstate, ngroups, chunk_size) != SSD_OK) {
        text = "rejected: " + g_detail;
        g_detail = saved;
        return text.c_str();
    }
    ssd::Dims d{batch, seqlen, nheads, headdim, dstate, ngroups, chunk_size,
                (seqlen + chunk_size - 1) / chunk_size};
    ssd::Args a;
    a.d = d;
    a.xdt = x_dtype;
    a.hprev_dt = x_dtype;
    char buf[512];
    if (ssd::use_fused(d, x_dtype) && ssd::pair_supported(d, x_dtype)) {
        const ssd::FusedSplit f = ssd::pair_split(d, ssd::device_sm_count());
        if (f.nseg > 1)
            snprintf(buf, sizeof buf,
                     "fused: k_ssd_pair x %lld CTAs (%lld whole (batch, head pair) slabs + the "
                     "last %lld pair slabs in %d segments of %lld tokens, after a states-only "
                     "pass and a combine), two heads per CTA, 128-token blocks, tcgen05 + TMA, "
                     "workspace %zu bytes",
                     (long long)(f.n_whole + f.tail * f.nseg), (long long)f.n_whole,
                     (long long)f.tail, f.nseg, (long long)f.seg_len, f.ws_bytes);
        else
            snprintf(buf, sizeof buf,
                     "fused: k_ssd_pair x %lld CTAs ((batch, head pair) slabs), two heads per "
                     "CTA, 128-token blocks, tcgen05 + TMA, no workspace",
                     (long long)(batch * nheads / 2));
    } else if (ssd::use_fused(d, x_dtype)) {
        const ssd::FusedSplit f = ssd::fused_split(d, ssd::device_sm_count());
        if (f.nseg > 1)
            snprintf(buf, sizeof buf,
                     "fused: k_ssd_fused x %lld CTAs (%lld whole (batch, head) slabs + the last "
                     "%lld slabs in %d segments of %lld tokens, after a states-only pass and a "
                     "combine), 128-token blocks, tcgen05 + TMA, workspace %zu bytes",
                     (long long)(f.n_whole + f.tail * f.nseg), (long long)f.n_whole,
                     (long long)f.tail, f.nseg, (long long)f.seg_len, f.ws_bytes);
        else
            snprintf(buf, sizeof buf,
                     "fused: k_ssd_fused x %lld CTAs ((batch, head) slabs), 128-token blocks, "
                     "tcgen05 + TMA, no workspace",
                     (long long)(batch * nheads));
    } else if (ssd::f32_split_plan(d, x_dtype)) {
        snprintf(buf, sizeof buf,
                 "staged: fp32 as bf16 hi + lo copies (k_split_hilo), chunk_cumsum simt, "
                 "chunk_state tcgen05 (k_chunk_state_tc_f32, three products), state_passing simt, "
                 "chunk_scan tcgen05 (k_chunk_scan_tc_f32, three products)");
    } else {
        snprintf(buf, sizeof buf,
                 "staged: chunk_cumsum simt, chunk_state %s, state_passing simt, chunk_scan %s",
                 ssd::uses_tc_chunk_state(a) ? "tcgen05" : "simt",
                 ssd::uses_tc_chunk_scan(a) ? "tcgen05" : "simt");
    }
    text = buf;
    return text.c_str();
}

ssd_status ssd_device_status(void *stream) {
    unsigned int *word = nullptr;
    ssd_status st;
    if ((st = cuda_status(ssd::device_error_word(&word), "device error word"))) return st;
    if ((st = cuda_status(cudaStreamSynchronize(static_cast<cudaStream_t>(stream)),
                          "stream synchronize")))
        return st;
    unsigned int v[2] = {0, 0};
    if ((st = cuda_status(cudaMemcpy(v, word, sizeof v, cudaMemcpyDeviceToHost), "read")))
        return st;
    if (v[0]) {
        const unsigned int zero[2] = {0, 0};
        if ((st = cuda_status(cudaMemcpy(word, zero, sizeof zero, cudaMemcpyHostToDevice),
                              "clear")))
            return st;
        if (v[0] & 4u) {
            static const char *const files[] = {"?", "ssd_fused.cu", "ssd_pair.cu", "ssd_tc.cu",
                                                "ssd_simt.cu", "ssd_selftest.cu", "ssd_tc_f32.cu"};
            const unsigned f = v[1] >> 16;
            return fail(SSD_ERR_DEVICE_BOUNDS,
                        "a device bounds check failed (flags 0x%x), first at %s line %u; the "
                        "access was skipped and outputs since the last check are not valid",
                        v[0], f < 7 ? files[f] : "?", v[1] & 0xffffu);
        }
        return fail(SSD_ERR_TIMEOUT, "a kernel gave up a bounded wait (flags 0x%x); outputs of "
                    "the calls since the last check are not valid", v[0]);
    }
    return ok();
}

ssd_status ssd_selftest_bounds_check(void *stream) {
    if (!ssd::bounds_checks_built())
        return fail(SSD_ERR_UNSUPPORTED, "bounds checks are compiled only into the debug build "
                    "(libssd_gb300_debug.so)");
    return cuda_status(ssd::launch_bounds_selftest(static_cast<cudaStream_t>(stream)),
                       "bounds self-test");
}

ssd_status ssd_selftest_wait_timeout(uint64_t limit_ns, void *stream) {
    if (limit_ns > 100000000ull)
        return fail(SSD_ERR_INVALID_ARG, "limit %llu ns above 100 ms", (unsigned long long)limit_ns);
    return cuda_status(ssd::launch_wait_selftest(limit_ns, static_cast<cudaStream_t>(stream)),
                       "wait self-test");
}

ssd_status ssd_workspace_size(int64_t batch, int64_t seqlen, int64_t nheads, int64_t headdim,
                              int64_t dstate, int64_t ngroups, int64_t chunk_size,
                              int32_t x_dtype, size_t *bytes) {
    if (!bytes) return fail(SSD_ERR_INVALID_ARG, "bytes: null pointer");
    *bytes = 0;
    if (x_dtype != SSD_F32 && x_dtype != SSD_BF16)
        return fail(SSD_ERR_INVALID_ARG, "x_dtype: unknown dtype code %d", x_dtype);
    ssd_status st = check_geometry(batch, seqlen, nheads, headdim, dstate, ngroups, chunk_size);
    if (st != SSD_OK) return st;
    ssd::Dims d{batch, seqlen, nheads, headdim, dstate, ngroups, chunk_size,
                (seqlen + chunk_size - 1) / chunk_size};
    *bytes = plan_workspace(d, x_dtype).total;
    return ok();
}

namespace {

// ssd_chunked_fwd (z = NULL) and ssd_chunked_fwd_gated.
ssd_status chunked_fwd_impl(const ssd_tensor *x, const ssd_tensor *dt, const ssd_tensor *A,
                            const ssd_tensor *Bm, const ssd_tensor *Cm, const ssd_tensor *D,
                            const ssd_tensor *z, const ssd_tensor *h0, int64_t chunk_size,
                            int64_t ngroups, ssd_tensor *y, ssd_tensor *final_states,
                            void *workspace, size_t workspace_bytes, void *stream) {
    if (!x) return fail(SSD_ERR_INVALID_ARG, "x: null tensor descriptor");
    if (x->ndim != 4) return fail(SSD_ERR_INVALID_ARG, "x: ndim %d, expected 4", x->ndim);
    if (!Bm) return fail(SSD_ERR_INVALID_ARG, "B: null tensor descriptor");
    if (Bm->ndim != 4) return fail(SSD_ERR_INVALID_ARG, "B: ndim %d, expected 4", Bm->ndim);
    const int64_t Bn = x->shape[0], L = x->shape[1], H = x->shape[2], P = x->shape[3];
    const int64_t N = Bm->shape[3], G = ngroups, Q = chunk_size;
    ssd_status st = check_geometry(Bn, L, H, P, N, G, Q);
    if (st != SSD_OK) return st;
    const int xdt = x->dtype;
    const int64_t sx[4] = {Bn, L, H, P}, sdt[3] = {Bn, L, H}, sh[1] = {H},
                  sbc[4] = {Bn, L, G, N}, sst[4] = {Bn, H, P, N};
    if ((st = check_tensor(x, "x", 4, sx, -1, false, true))) return st;
    if ((st = check_tensor(dt, "dt", 3, sdt, SSD_F32, false, false))) return st;
    if ((st = check_tensor(A, "A", 1, sh, SSD_F32, true, false))) return st;
    if ((st = check_tensor(Bm, "B", 4, sbc, xdt, false, true))) return st;
    if ((st = check_tensor(Cm, "C", 4, sbc, xdt, false, true))) return st;
    if (D && (st = check_tensor(D, "D", 1, sh, SSD_F32, true, false))) return st;
    if (h0 && (st = check_tensor(h0, "initial_states", 4, sst, SSD_F32, true, true))) return st;
    if (z && (st = check_tensor(z, "z", 4, sx, xdt, false, true))) return st;
    if ((st = check_tensor(y, "y", 4, sx, xdt, false, true))) return st;
    if (final_states &&
        (st = check_tensor(final_states, "final_states", 4, sst, SSD_F32, true, true)))
        return st;

    ssd::Dims d{Bn, L, H, P, N, G, Q, (L + Q - 1) / Q};
    const Plan plan = plan_workspace(d, xdt);
    if (Bn > 0 && plan.total > 0) {
        if (workspace_bytes < plan.total)
            return fail(SSD_ERR_WORKSPACE, "workspace %zu bytes, need %zu", workspace_bytes,
                        plan.total);
        if (!workspace) return fail(SSD_ERR_WORKSPACE, "workspace: null pointer");
        if (reinterpret_cast<uintptr_t>(workspace) % 256)
            return fail(SSD_ERR_ALIGNMENT, "workspace %p not 256-byte aligned", workspace);
    }

    const Range ins[] = {range_of(x), range_of(dt), range_of(A), range_of(Bm), range_of(Cm),
                         range_of(D), range_of(h0), range_of(z)};
    const char *in_names[] = {"x", "dt", "A", "B", "C", "D", "initial_states", "z"};
    const Range ry = range_of(y), rf = range_of(final_states);
    const Range rw = range_raw(workspace, Bn > 0 ? plan.total : 0);
    for (int i = 0; i < 8; ++i) {
        if (overlap(ry, ins[i])) return fail(SSD_ERR_INVALID_ARG, "y overlaps %s", in_names[i]);
        if (overlap(rf, ins[i]))
            return fail(SSD_ERR_INVALID_ARG, "final_states overlaps %s", in_names[i]);
        if (overlap(rw, ins[i]))
            return fail(SSD_ERR_INVALID_ARG, "workspace overlaps %s", in_names[i]);
    }
    if (overlap(ry, rf)) return fail(SSD_ERR_INVALID_ARG, "y overlaps final_states");
    if (overlap(rw, ry) || overlap(rw, rf))
        return fail(SSD_ERR_INVALID_ARG, "workspace overlaps an output");
    if (Bn == 0) return ok();
    auto dp = [](const ssd_tensor *t) -> const void * { return t ? t->data : nullptr; };
    if ((st = check_device_ptrs({{dp(x), "x"}, {dp(dt), "dt"}, {dp(A), "A"}, {dp(Bm), "B"},
                                 {dp(Cm), "C"}, {dp(D), "D"}, {dp(h0), "initial_states"},
                                 {dp(z), "z"}, {dp(y), "y"}, {dp(final_states), "final_states"},
                                 {workspace, "workspace"}})))
        return st;

    ssd::Args a;
    a.d = d;
    a.xdt = xdt;
    fill_x(a, x);
    fill_dt(a, dt);
    a.A = static_cast<const float *>(A->data);
    a.D = D ? static_cast<const float *>(D->data) : nullptr;
    fill_bc(a, Bm, Cm);
    a.h0 = h0 ? static_cast<const float *>(h0->data) : nullptr;
    fill_y(a, y);
    a.final_states = final_states ? static_cast<float *>(final_states->data) : nullptr;
    if (z) {
        a.z = z->data;
        a.z_sb = z->stride[0];
        a.z_sl = z->stride[1];
        a.z_sh = z->stride[2];
    }
    char *ws = static_cast<char *>(workspace);
    a.G = reinterpret_cast<float *>(ws + plan.off_G);
    a.S = reinterpret_cast<float *>(ws + plan.off_S);
    a.h_prev = ws + plan.off_hp;
    a.hprev_dt = xdt;
    a.ws = ws;
    if (plan.f32_split) {
        a.f32_split = true;
        a.f32s = {ws + plan.off_x_hi, ws + plan.off_x_lo, ws + plan.off_b_hi, ws + plan.off_b_lo,
                  ws + plan.off_c_hi, ws + plan.off_c_lo, ws + plan.off_hp_hi, ws + plan.off_hp_lo};
    }

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (plan.fused) {
        if ((st = cuda_status(ssd::pair_supported(a.d, xdt) ? ssd::launch_pair(a, s)
                                                             : ssd::launch_fused(a, s),
                              "fused forward")))
            return st;
        if (z && (st = cuda_status(ssd::launch_gate(a, s), "output gate"))) return st;
        return ok();
    }
    if (L > 0) {
        if (a.f32_split && (st = cuda_status(ssd::split_inputs_f32(a, s), "fp32 hi/lo split")))
            return st;
        if ((st = cuda_status(ssd::launch_chunk_cumsum(a, s), "chunk_cumsum"))) return st;
        if ((st = cuda_status(ssd::launch_chunk_state(a, s), "chunk_state"))) return st;
    }
    if ((st = cuda_status(ssd::launch_state_passing(a, s), "state_passing"))) return st;
    if (L > 0 && (st = cuda_status(ssd::launch_chunk_scan(a, s), "chunk_scan"))) return st;
    if (z && L > 0 && (st = cuda_status(ssd::launch_gate(a, s), "output gate"))) return st;
    return ok();
}

}  // namespace

ssd_status ssd_chunked_fwd(const ssd_tensor *x, const ssd_tensor *dt, const ssd_tensor *A,
                           const ssd_tensor *Bm, const ssd_tensor *Cm, const ssd_tensor *D,
                           const ssd_tensor *h0, int64_t chunk_size, int64_t ngroups,
                           ssd_tensor *y, ssd_tensor *final_states, void *workspace,
                           size_t workspace_bytes, void *stream) {
    return chunked_fwd_impl(x, dt, A, Bm, Cm, D, nullptr, h0, chunk_size, ngroups, y,
                            final_states, workspace, workspace_bytes, stream);
}

ssd_status ssd_chunked_fwd_gated(const ssd_tensor *x, const ssd_tensor *dt, const ssd_tensor *A,
                                 const ssd_tensor *Bm, const ssd_tensor *Cm, const ssd_tensor *D,
                                 const ssd_tensor *z, const ssd_tensor *h0, int64_t chunk_size,
                                 int64_t ngroups, ssd_tensor *y, ssd_tensor *final_states,
                                 void *workspace, size_t workspace_bytes, void *stream) {
    if (!z) return fail(SSD_ERR_INVALID_ARG, "z: null tensor descriptor");
    return chunked_fwd_impl(x, dt, A, Bm, Cm, D, z, h0, chunk_size, ngroups, y, final_states,
                            workspace, workspace_bytes, stream);
}

namespace {

// ssd_state_update (tokens = false: no token axis, T = 1) and
// ssd_state_update_tokens (tokens = true).
ssd_status state_update_impl(bool tokens, ssd_tensor *state, const ssd_tensor *x,
                             const ssd_tensor *dt, const ssd_tensor *A, const ssd_tensor *Bm,
                             const ssd_tensor *Cm, const ssd_tensor *D, const ssd_tensor *z,
                             const ssd_tensor *dt_bias, int32_t dt_softplus, int64_t ngroups,
                             ssd_tensor *out, ssd_tensor *inter, const ssd_tensor *parent,
                             const ssd_tensor *slots, int32_t update_state, void *stream) {
    if (!state) return fail(SSD_ERR_INVALID_ARG, "state: null tensor descriptor");
    if (state->ndim != 4) return fail(SSD_ERR_INVALID_ARG, "state: ndim %d, expected 4",
                                      state->ndim);
    if (!x) return fail(SSD_ERR_INVALID_ARG, "x: null tensor descriptor");
    if (tokens && x->ndim != 4)
        return fail(SSD_ERR_INVALID_ARG, "x: ndim %d, expected 4", x->ndim);
    // rows come from x; the state holds one entry per row, or a pool of S
    // slots addressed through `slots`
    const int64_t Bn = x->shape[0], S = state->shape[0], H = state->shape[1],
                  P = state->shape[2], N = state->shape[3], G = ngroups,
                  T = tokens ? x->shape[1] : 1;
    if (Bn < 0 || T < 0 || S < 0)
        return fail(SSD_ERR_INVALID_ARG, "batch %lld / tokens %lld / state slots %lld negative",
                    (long long)Bn, (long long)T, (long long)S);
    if (!slots && S != Bn)
        return fail(SSD_ERR_INVALID_ARG, "state: shape[0] = %lld, expected the batch %lld (or "
                    "give state_indices)", (long long)S, (long long)Bn);
    if (slots && S > (int64_t(1) << 31) - 1)
        return fail(SSD_ERR_UNSUPPORTED, "state pool of %lld slots above 2^31 - 1", (long long)S);
    if (H <= 0 || G <= 0) return fail(SSD_ERR_INVALID_ARG, "nheads %lld / ngroups %lld must be "
                                      "positive", (long long)H, (long long)G);
    if (H % G) return fail(SSD_ERR_INVALID_ARG, "nheads %lld is not a multiple of ngroups %lld",
                           (long long)H, (long long)G);
    if (!supported_dim(P))
        return fail(SSD_ERR_UNSUPPORTED, "headdim %lld unsupported (16, 32, 64 or 128)",
                    (long long)P);
    if (!supported_dim(N))
        return fail(SSD_ERR_UNSUPPORTED, "dstate %lld unsupported (16, 32, 64 or 128)",
                    (long long)N);
    if (Bn > 65535 || H > 65535 || T > (int64_t(1) << 30))
        return fail(SSD_ERR_UNSUPPORTED, "batch %lld or nheads %lld above 65535, or tokens %lld "
                    "above 2^30", (long long)Bn, (long long)H, (long long)T);
    if (parent && !inter)
        return fail(SSD_ERR_INVALID_ARG, "parent needs intermediate_states (the parents' "
                    "states are read from there)");
    const int xdt = x->dtype;
    // shapes with the token axis (index 1) when `tokens`, without it otherwise
    const int k = tokens ? 1 : 0;
    const int64_t sst[4] = {S, H, P, N};
    const int64_t sx4[4] = {Bn, T, H, P}, sx3[3] = {Bn, H, P};
    const int64_t sdt3[3] = {Bn, T, H}, sdt2[2] = {Bn, H};
    const int64_t sbc4[4] = {Bn, T, G, N}, sbc3[3] = {Bn, G, N};
    const int64_t sh[1] = {H}, sin[5] = {S, T, H, P, N}, spar[2] = {Bn, T}, sslot[1] = {Bn};
    const int64_t *sx = tokens ? sx4 : sx3, *sdt = tokens ? sdt3 : sdt2,
                  *sbc = tokens ? sbc4 : sbc3;
    ssd_status st;
    // the state is kept in f32 or bf16; its cache in the same dtype
    if ((st = check_tensor(state, "state", 4, sst, -1, true, true))) return st;
    if ((st = check_tensor(x, "x", 3 + k, sx, -1, false, false))) return st;
    if ((st = check_tensor(dt, "dt", 2 + k, sdt, SSD_F32, false, false))) return st;
    if ((st = check_tensor(A, "A", 1, sh, SSD_F32, true, false))) return st;
    if ((st = check_tensor(Bm, "B", 3 + k, sbc, xdt, false, true))) return st;
    if ((st = check_tensor(Cm, "C", 3 + k, sbc, xdt, false, true))) return st;
    for (int i = 0; i < 2 + k; ++i)
        if (Bm->stride[i] != Cm->stride[i])
            return fail(SSD_ERR_INVALID_ARG, "B and C must have the same strides");
    if (D && (st = check_tensor(D, "D", 1, sh, SSD_F32, true, false))) return st;
    if (z && (st = check_tensor(z, "z", 3 + k, sx, xdt, false, false))) return st;
    if (dt_bias && (st = check_tensor(dt_bias, "dt_bias", 1, sh, SSD_F32, true, false))) return st;
    if ((st = check_tensor(out, "out", 3 + k, sx, xdt, false, false))) return st;
    if (inter &&
        (st = check_tensor(inter, "intermediate_states", 5, sin, state->dtype, true, true)))
        return st;
    if (parent && (st = check_tensor(parent, "parent", 2, spar, SSD_I32, false, false)))
        return st;
    if (slots && (st = check_tensor(slots, "state_indices", 1, sslot, SSD_I32, true, false)))
        return st;

    const Range ins[] = {range_of(x),  range_of(dt), range_of(A),       range_of(Bm),
                         range_of(Cm), range_of(D),  range_of(z),       range_of(dt_bias),
                         range_of(parent), range_of(slots)};
    const char *in_names[] = {"x", "dt", "A", "B", "C", "D", "z", "dt_bias", "parent",
                              "state_indices"};
    const Range rs = range_of(state), ro = range_of(out), ri = range_of(inter);
    for (int i = 0; i < 10; ++i) {
        if (overlap(ro, ins[i])) return fail(SSD_ERR_INVALID_ARG, "out overlaps %s", in_names[i]);
        if (overlap(rs, ins[i]))
            return fail(SSD_ERR_INVALID_ARG, "state overlaps %s", in_names[i]);
        if (overlap(ri, ins[i]))
            return fail(SSD_ERR_INVALID_ARG, "intermediate_states overlaps %s", in_names[i]);
    }
    if (overlap(ro, rs)) return fail(SSD_ERR_INVALID_ARG, "out overlaps state");
    if (overlap(ri, rs) || overlap(ri, ro))
        return fail(SSD_ERR_INVALID_ARG, "intermediate_states overlaps state or out");
    if (Bn == 0 || T == 0) return ok();
    auto dp = [](const ssd_tensor *t) -> const void * { return t ? t->data : nullptr; };
    if ((st = check_device_ptrs({{dp(state), "state"}, {dp(x), "x"}, {dp(dt), "dt"},
                                 {dp(A), "A"}, {dp(Bm), "B"}, {dp(Cm), "C"}, {dp(D), "D"},
                                 {dp(z), "z"}, {dp(dt_bias), "dt_bias"}, {dp(out), "out"},
                                 {dp(inter), "intermediate_states"}, {dp(parent), "parent"},
                                 {dp(slots), "state_indices"}})))
        return st;

    // stride of the token axis (0 without one) and of the axes after it
    auto sT = [&](const ssd_tensor *t) -> int64_t { return tokens ? t->stride[1] : 0; };
    auto sAt = [&](const ssd_tensor *t, int i) -> int64_t { return t->stride[i + k]; };
    ssd::SsuArgs a;
    a.B = int(Bn);
    a.T = int(T);
    a.H = int(H);
    a.P = int(P);
    a.N = int(N);
    a.G = int(G);
    a.xdt = xdt;
    a.softplus = dt_softplus ? 1 : 0;
    a.update = update_state ? 1 : 0;
    a.sdt = state->dtype == SSD_BF16 ? ssd::DT_BF16 : ssd::DT_F32;
    a.state = state->data;
    a.x = x->data;
    a.x_sb = x->stride[0];
    a.x_st = sT(x);
    a.x_sh = sAt(x, 1);
    a.dt = static_cast<const float *>(dt->data);
    a.dt_sb = dt->stride[0];
    a.dt_st = sT(dt);
    a.A = static_cast<const float *>(A->data);
    a.D = D ? static_cast<const float *>(D->data) : nullptr;
    a.dt_bias = dt_bias ? static_cast<const float *>(dt_bias->data) : nullptr;
    a.Bm = Bm->data;
    a.Cm = Cm->data;
    a.bc_sb = Bm->stride[0];
    a.bc_st = sT(Bm);
    a.bc_sg = sAt(Bm, 1);
    a.z = z ? z->data : nullptr;
    a.z_sb = z ? z->stride[0] : 0;
    a.z_st = z ? sT(z) : 0;
    a.z_sh = z ? sAt(z, 1) : 0;
    a.out = out->data;
    a.o_sb = out->stride[0];
    a.o_st = sT(out);
    a.o_sh = sAt(out, 1);
    a.inter = inter ? inter->data : nullptr;
    a.parent = parent ? static_cast<const int32_t *>(parent->data) : nullptr;
    a.par_sb = parent ? parent->stride[0] : 0;
    a.slots = slots ? static_cast<const int32_t *>(slots->data) : nullptr;
    a.S = int(S);
    return cuda_status(ssd::launch_ssu(a, static_cast<cudaStream_t>(stream)), "state update");
}

}  // namespace

ssd_status ssd_state_update(ssd_tensor *state, const ssd_tensor *x, const ssd_tensor *dt,
                            const ssd_tensor *A, const ssd_tensor *Bm, const ssd_tensor *Cm,
                            const ssd_tensor *D, const ssd_tensor *z, const ssd_tensor *dt_bias,
                            int32_t dt_softplus, int64_t ngroups, ssd_tensor *out, void *stream) {
    return state_update_impl(false, state, x, dt, A, Bm, Cm, D, z, dt_bias, dt_softplus, ngroups,
                             out, nullptr, nullptr, nullptr, 1, stream);
}

ssd_status ssd_state_update_tokens(ssd_tensor *state, const ssd_tensor *x, const ssd_tensor *dt,
                                   const ssd_tensor *A, const ssd_tensor *Bm,
                                   const ssd_tensor *Cm, const ssd_tensor *D, const ssd_tensor *z,
                                   const ssd_tensor *dt_bias, int32_t dt_softplus,
                                   int64_t ngroups, ssd_tensor *out,
                                   ssd_tensor *intermediate_states, const ssd_tensor *parent,
                                   const ssd_tensor *state_indices, int32_t update_state,
                                   void *stream) {
    return state_update_impl(true, state, x, dt, A, Bm, Cm, D, z, dt_bias, dt_softplus, ngroups,
                             out, intermediate_states, parent, state_indices, update_state,
                             stream);
}

ssd_status ssd_mixer_prologue(const ssd_tensor *xBC, const ssd_tensor *conv_weight,
                              const ssd_tensor *conv_bias, ssd_tensor *conv_state,
                              ssd_tensor *conv_windows, const ssd_tensor *conv_state_indices,
                              const ssd_tensor *dt,
                              const ssd_tensor *dt_bias, int32_t dt_softplus, int64_t ngroups,
                              ssd_tensor *x, ssd_tensor *Bm, ssd_tensor *Cm, ssd_tensor *dt_out,
                              void *stream) {
    if (!xBC || !x || !Bm || !conv_weight)
        return fail(SSD_ERR_INVALID_ARG, "xBC / conv_weight / x / B: null tensor descriptor");
    if (xBC->ndim != 3) return fail(SSD_ERR_INVALID_ARG, "xBC: ndim %d, expected 3", xBC->ndim);
    if (x->ndim != 4 || Bm->ndim != 4)
        return fail(SSD_ERR_INVALID_ARG, "x / B: ndim must be 4");
    if (conv_weight->ndim != 2)
        return fail(SSD_ERR_INVALID_ARG, "conv_weight: ndim %d, expected 2", conv_weight->ndim);
    const int64_t Bn = xBC->shape[0], L = xBC->shape[1], Dc = xBC->shape[2];
    const int64_t H = x->shape[2], P = x->shape[3], N = Bm->shape[3], G = ngroups,
                  W = conv_weight->shape[1];
    if (Bn < 0 || L < 0) return fail(SSD_ERR_INVALID_ARG, "negative batch or seqlen");
    if (H <= 0 || G <= 0)
        return fail(SSD_ERR_INVALID_ARG, "nheads %lld / ngroups %lld must be positive",
                    (long long)H, (long long)G);
    if (!supported_dim(P) || !supported_dim(N))
        return fail(SSD_ERR_UNSUPPORTED, "headdim %lld / dstate %lld unsupported (16, 32, 64 or "
                    "128)", (long long)P, (long long)N);
    if (Dc != H * P + 2 * G * N)
        return fail(SSD_ERR_INVALID_ARG, "xBC has %lld channels; nheads * headdim + 2 * ngroups * "
                    "dstate = %lld", (long long)Dc, (long long)(H * P + 2 * G * N));
    if (W < 1 || W > 4)
        return fail(SSD_ERR_UNSUPPORTED, "conv width %lld unsupported (1 to 4)", (long long)W);
    if (Bn > 65535 || (L + 63) / 64 > 65535)
        return fail(SSD_ERR_UNSUPPORTED, "batch %lld above 65535 or seqlen %lld above 4194240",
                    (long long)Bn, (long long)L);
    const int xdt = xBC->dtype;
    // with slot indices the conv state and windows are pools of S slots
    if (conv_state_indices && !conv_state)
        return fail(SSD_ERR_INVALID_ARG, "conv_state_indices needs conv_state (the slot pool)");
    const int64_t S = conv_state_indices ? conv_state->shape[0] : Bn;
    if (S < 0 || S > (int64_t(1) << 31) - 1)
        return fail(SSD_ERR_INVALID_ARG, "conv_state: %lld slots", (long long)S);
    const int64_t sin[3] = {Bn, L, Dc}, sw[2] = {Dc, W}, sb[1] = {Dc}, sst[3] = {S, Dc, W},
                  swin[4] = {S, L, Dc, W}, sdt[3] = {Bn, L, H}, sh[1] = {H},
                  sx[4] = {Bn, L, H, P}, sbc[4] = {Bn, L, G, N}, sslot[1] = {Bn};
    ssd_status st;
    if ((st = check_tensor(xBC, "xBC", 3, sin, -1, false, true))) return st;
    if ((st = check_tensor(conv_weight, "conv_weight", 2, sw, SSD_F32, true, false))) return st;
    if (conv_bias && (st = check_tensor(conv_bias, "conv_bias", 1, sb, SSD_F32, true, false)))
        return st;
    if (conv_state && (st = check_tensor(conv_state, "conv_state", 3, sst, xdt, true, false)))
        return st;
    if (conv_windows &&
        (st = check_tensor(conv_windows, "conv_windows", 4, swin, xdt, true, false)))
        return st;
    if ((st = check_tensor(dt, "dt", 3, sdt, SSD_F32, false, false))) return st;
    if (dt_bias && (st = check_tensor(dt_bias, "dt_bias", 1, sh, SSD_F32, true, false))) return st;
    if ((st = check_tensor(x, "x", 4, sx, xdt, false, true))) return st;
    if ((st = check_tensor(Bm, "B", 4, sbc, xdt, false, true))) return st;
    if ((st = check_tensor(Cm, "C", 4, sbc, xdt, false, true))) return st;
    if ((st = check_tensor(dt_out, "dt_out", 3, sdt, SSD_F32, false, false))) return st;
    if (conv_state_indices && (st = check_tensor(conv_state_indices, "conv_state_indices", 1,
                                                 sslot, SSD_I32, true, false)))
        return st;

    // every output against every input and each other; the conv state is
    // updated in place, so it may overlap nothing else
    const Range ins[] = {range_of(xBC), range_of(conv_weight), range_of(conv_bias),
                         range_of(dt), range_of(dt_bias), range_of(conv_state_indices)};
    const char *in_names[] = {"xBC", "conv_weight", "conv_bias", "dt", "dt_bias",
                              "conv_state_indices"};
    const Range outs[] = {range_of(x), range_of(Bm), range_of(Cm), range_of(dt_out),
                          range_of(conv_state), range_of(conv_windows)};
    const char *out_names[] = {"x", "B", "C", "dt_out", "conv_state", "conv_windows"};
    for (int o = 0; o < 6; ++o) {
        for (int i = 0; i < 6; ++i)
            if (overlap(outs[o], ins[i]))
                return fail(SSD_ERR_INVALID_ARG, "%s overlaps %s", out_names[o], in_names[i]);
        for (int o2 = o + 1; o2 < 6; ++o2)
            if (overlap(outs[o], outs[o2]))
                return fail(SSD_ERR_INVALID_ARG, "%s overlaps %s", out_names[o], out_names[o2]);
    }
    if (Bn == 0 || L == 0) return ok();
    auto dp = [](const ssd_tensor *t) -> const void * { return t ? t->data : nullptr; };
    if ((st = check_device_ptrs({{dp(xBC), "xBC"}, {dp(conv_weight), "conv_weight"},
                                 {dp(conv_bias), "conv_bias"}, {dp(conv_state), "conv_state"},
                                 {dp(conv_windows), "conv_windows"}, {dp(dt), "dt"},
                                 {dp(dt_bias), "dt_bias"}, {dp(x), "x"}, {dp(Bm), "B"},
                                 {dp(Cm), "C"}, {dp(dt_out), "dt_out"},
                                 {dp(conv_state_indices), "conv_state_indices"}})))
        return st;
    ssd::MixerArgs a;
    a.B = int(Bn);
    a.L = L;
    a.H = int(H);
    a.P = int(P);
    a.G = int(G);
    a.N = int(N);
    a.Dc = int(Dc);
    a.W = int(W);
    a.xdt = xdt;
    a.softplus = dt_softplus ? 1 : 0;
    a.xBC = xBC->data;
    a.in_sb = xBC->stride[0];
    a.in_sl = xBC->stride[1];
    a.conv_w = static_cast<const float *>(conv_weight->data);
    a.conv_b = conv_bias ? static_cast<const float *>(conv_bias->data) : nullptr;
    a.state = conv_state ? conv_state->data : nullptr;
    a.windows = conv_windows ? conv_windows->data : nullptr;
    a.slots = conv_state_indices ? static_cast<const int32_t *>(conv_state_indices->data)
                                 : nullptr;
    a.S = int(S);
    a.dt = static_cast<const float *>(dt->data);
    a.dt_sb = dt->stride[0];
    a.dt_sl = dt->stride[1];
    a.dt_bias = dt_bias ? static_cast<const float *>(dt_bias->data) : nullptr;
    a.dt_out = static_cast<float *>(dt_out->data);
    a.do_sb = dt_out->stride[0];
    a.do_sl = dt_out->stride[1];
    a.x = x->data;
    a.x_sb = x->stride[0];
    a.x_sl = x->stride[1];
    a.x_sh = x->stride[2];
    a.Bo = Bm->data;
    a.b_sb = Bm->stride[0];
    a.b_sl = Bm->stride[1];
    a.b_sg = Bm->stride[2];
    a.Co = Cm->data;
    a.c_sb = Cm->stride[0];
    a.c_sl = Cm->stride[1];
    a.c_sg = Cm->stride[2];
    return cuda_status(ssd::launch_mixer_prologue(a, static_cast<cudaStream_t>(stream)),
                       "mixer prologue");
}

ssd_status ssd_stage_chunk_cumsum(const ssd_tensor *dt, const ssd_tensor *A, int64_t chunk_size,
                                  ssd_tensor *G, void *stream) {
    if (!dt) return fail(SSD_ERR_INVALID_ARG, "dt: null tensor descriptor");
    if (dt->ndim != 3) return fail(SSD_ERR_INVALID_ARG, "dt: ndim %d, expected 3", dt->ndim);
    const int64_t Bn = dt->shape[0], L = dt->shape[1], H = dt->shape[2], Q = chunk_size;
    ssd_status st = check_geometry(Bn, L, H, 64, 64, 1, Q);
    if (st != SSD_OK) return st;
    const int64_t nc = (L + Q - 1) / Q;
    const int64_t sdt[3] = {Bn, L, H}, sh[1] = {H}, sg[3] = {Bn, H, nc * Q};
    if ((st = check_tensor(dt, "dt", 3, sdt, SSD_F32, false, false))) return st;
    if ((st = check_tensor(A, "A", 1, sh, SSD_F32, true, false))) return st;
    if ((st = check_tensor(G, "G", 3, sg, SSD_F32, true, false))) return st;
    if (overlap(range_of(G), range_of(dt)) || overlap(range_of(G), range_of(A)))
        return fail(SSD_ERR_INVALID_ARG, "G overlaps an input");
    if (Bn == 0 || L == 0) return ok();
    if ((st = check_device_ptrs({{dt->data, "dt"}, {A->data, "A"}, {G->data, "G"}}))) return st;
    ssd::Args a;
    a.d = ssd::Dims{Bn, L, H, 64, 64, 1, Q, nc};
    fill_dt(a, dt);
    a.A = static_cast<const float *>(A->data);
    a.G = static_cast<float *>(G->data);
    if ((st = cuda_status(ssd::launch_chunk_cumsum(a, static_cast<cudaStream_t>(stream)),
                          "chunk_cumsum")))
        return st;
    return ok();
}

ssd_status ssd_stage_chunk_state(const ssd_tensor *x, const ssd_tensor *Bm, const ssd_tensor *dt,
                                 const ssd_tensor *G, int64_t chunk_size, int64_t ngroups,
                                 ssd_tensor *S, void *stream) {
    if (!x || !Bm) return fail(SSD_ERR_INVALID_ARG, "x / B: null tensor descriptor");
    if (x->ndim != 4 || Bm->ndim != 4) return fail(SSD_ERR_INVALID_ARG, "x / B: ndim must be 4");
    const int64_t Bn = x->shape[0], L = x->shape[1], H = x->shape[2], P = x->shape[3];
    const int64_t N = Bm->shape[3], Gn = ngroups, Q = chunk_size;
    ssd_status st = check_geometry(Bn, L, H, P, N, Gn, Q);
    if (st != SSD_OK) return st;
    const int64_t nc = (L + Q - 1) / Q;
    const int64_t sx[4] = {Bn, L, H, P}, sdt[3] = {Bn, L, H}, sbc[4] = {Bn, L, Gn, N},
                  sg[3] = {Bn, H, nc * Q}, ss[5] = {Bn, nc, H, P, N};
    if ((st = check_tensor(x, "x", 4, sx, -1, false, true))) return st;
    if ((st = check_tensor(Bm, "B", 4, sbc, x->dtype, false, true))) return st;
    if ((st = check_tensor(dt, "dt", 3, sdt, SSD_F32, false, false))) return st;
    if ((st = check_tensor(G, "G", 3, sg, SSD_F32, true, false))) return st;
    if ((st = check_tensor(S, "S", 5, ss, SSD_F32, true, true))) return st;
    const Range rs = range_of(S);
    if (overlap(rs, range_of(x)) || overlap(rs, range_of(Bm)) || overlap(rs, range_of(dt)) ||
        overlap(rs, range_of(G)))
        return fail(SSD_ERR_INVALID_ARG, "S overlaps an input");
    if (Bn == 0 || L == 0) return ok();
    if ((st = check_device_ptrs({{x->data, "x"}, {Bm->data, "B"}, {dt->data, "dt"},
                                 {G->data, "G"}, {S->data, "S"}})))
        return st;
    ssd::Args a;
    a.d = ssd::Dims{Bn, L, H, P, N, Gn, Q, nc};
    a.xdt = x->dtype;
    fill_x(a, x);
    fill_bc(a, Bm, nullptr);
    fill_dt(a, dt);
    a.G = static_cast<float *>(G->data);
    a.S = static_cast<float *>(S->data);
    if ((st = cuda_status(ssd::launch_chunk_state(a, static_cast<cudaStream_t>(stream)),
                          "chunk_state")))
        return st;
    return ok();
}

ssd_status ssd_stage_state_passing(const ssd_tensor *S, const ssd_tensor *G,
                                   const ssd_tensor *h0, int64_t chunk_size, ssd_tensor *h_prev,
                                   ssd_tensor *final_states, void *stream) {
    if (!S) return fail(SSD_ERR_INVALID_ARG, "S: null tensor descriptor");
    if (S->ndim != 5) return fail(SSD_ERR_INVALID_ARG, "S: ndim %d, expected 5", S->ndim);
    if (!G || G->ndim != 3) return fail(SSD_ERR_INVALID_ARG, "G: missing or ndim != 3");
    const int64_t Bn = S->shape[0], nc = S->shape[1], H = S->shape[2], P = S->shape[3],
                  N = S->shape[4], Q = chunk_size;
    ssd_status st = check_geometry(Bn, nc * Q, H, P, N, 1, Q);
    if (st != SSD_OK) return st;
    const int64_t ss[5] = {Bn, nc, H, P, N}, sg[3] = {Bn, H, nc * Q}, sst[4] = {Bn, H, P, N};
    if ((st = check_tensor(S, "S", 5, ss, SSD_F32, true, true))) return st;
    if ((st = check_tensor(G, "G", 3, sg, SSD_F32, true, false))) return st;
    if (h0 && (st = check_tensor(h0, "initial_states", 4, sst, SSD_F32, true, true))) return st;
    if ((st = check_tensor(h_prev, "h_prev", 5, ss, -1, true, true))) return st;
    if (final_states &&
        (st = check_tensor(final_states, "final_states", 4, sst, SSD_F32, true, true)))
        return st;
    const Range rh = range_of(h_prev), rf = range_of(final_states);
    const Range ins[] = {range_of(S), range_of(G), range_of(h0)};
    for (const Range &r : ins)
        if (overlap(rh, r) || overlap(rf, r))
            return fail(SSD_ERR_INVALID_ARG, "an output overlaps an input");
    if (overlap(rh, rf)) return fail(SSD_ERR_INVALID_ARG, "h_prev overlaps final_states");
    if (Bn == 0) return ok();
    if ((st = check_device_ptrs({{S->data, "S"}, {G->data, "G"},
                                 {h0 ? h0->data : nullptr, "initial_states"},
                                 {h_prev->data, "h_prev"},
                                 {final_states ? final_states->data : nullptr, "final_states"}})))
        return st;
    ssd::Args a;
    a.d = ssd::Dims{Bn, nc * Q, H, P, N, 1, Q, nc};
    a.S = static_cast<float *>(S->data);
    a.G = static_cast<float *>(G->data);
    a.h0 = h0 ? static_cast<const float *>(h0->data) : nullptr;
    a.h_prev = h_prev->data;
    a.hprev_dt = h_prev->dtype;
    a.final_states = final_states ? static_cast<float *>(final_states->data) : nullptr;
    if ((st = cuda_status(ssd::launch_state_passing(a, static_cast<cudaStream_t>(stream)),
                          "state_passing")))
        return st;
    return ok();
}

ssd_status ssd_stage_chunk_scan(const ssd_tensor *x, const ssd_tensor *dt, const ssd_tensor *G,
                                const ssd_tensor *Bm, const ssd_tensor *Cm, const ssd_tensor *D,
                                const ssd_tensor *h_prev, int64_t chunk_size, int64_t ngroups,
                                ssd_tensor *y, void *stream) {
    if (!x || !Bm) return fail(SSD_ERR_INVALID_ARG, "x / B: null tensor descriptor");
    if (x->ndim != 4 || Bm->ndim != 4) return fail(SSD_ERR_INVALID_ARG, "x / B: ndim must be 4");
    const int64_t Bn = x->shape[0], L = x->shape[1], H = x->shape[2], P = x->shape[3];
    const int64_t N = Bm->shape[3], Gn = ngroups, Q = chunk_size;
    ssd_status st = check_geometry(Bn, L, H, P, N, Gn, Q);
    if (st != SSD_OK) return st;
    const int64_t nc = (L + Q - 1) / Q;
    const int xdt = x->dtype;
    const int64_t sx[4] = {Bn, L, H, P}, sdt[3] = {Bn, L, H}, sbc[4] = {Bn, L, Gn, N},
                  sg[3] = {Bn, H, nc * Q}, ss[5] = {Bn, nc, H, P, N}, sh[1] = {H};
    if ((st = check_tensor(x, "x", 4, sx, -1, false, true))) return st;
    if ((st = check_tensor(dt, "dt", 3, sdt, SSD_F32, false, false))) return st;
    if ((st = check_tensor(G, "G", 3, sg, SSD_F32, true, false))) return st;
    if ((st = check_tensor(Bm, "B", 4, sbc, xdt, false, true))) return st;
    if ((st = check_tensor(Cm, "C", 4, sbc, xdt, false, true))) return st;
    if (D && (st = check_tensor(D, "D", 1, sh, SSD_F32, true, false))) return st;
    if ((st = check_tensor(h_prev, "h_prev", 5, ss, xdt, true, true))) return st;
    if ((st = check_tensor(y, "y", 4, sx, xdt, false, true))) return st;
    const Range ry = range_of(y);
    const Range ins[] = {range_of(x), range_of(dt), range_of(G), range_of(Bm),
                         range_of(Cm), range_of(D), range_of(h_prev)};
    for (const Range &r : ins)
        if (overlap(ry, r)) return fail(SSD_ERR_INVALID_ARG, "y overlaps an input");
    if (Bn == 0 || L == 0) return ok();
    if ((st = check_device_ptrs({{x->data, "x"}, {dt->data, "dt"}, {G->data, "G"},
                                 {Bm->data, "B"}, {Cm->data, "C"}, {D ? D->data : nullptr, "D"},
                                 {h_prev->data, "h_prev"}, {y->data, "y"}})))
        return st;
    ssd::Args a;
    a.d = ssd::Dims{Bn, L, H, P, N, Gn, Q, nc};
    a.xdt = xdt;
    fill_x(a, x);
    fill_dt(a, dt);
    a.G = static_cast<float *>(G->data);
    fill_bc(a, Bm, Cm);
    a.D = D ? static_cast<const float *>(D->data) : nullptr;
    a.h_prev = h_prev->data;
    a.hprev_dt = xdt;
    fill_y(a, y);
    if ((st = cuda_status(ssd::launch_chunk_scan(a, static_cast<cudaStream_t>(stream)),
                          "chunk_scan")))
        return st;
    return ok();
}

}  // extern "C"

/* ---- sequence sharding over ranks ---------------------------------------- */

namespace ssd {
cudaError_t launch_segment_logdecay(const float *dt, int64_t dt_sb, int64_t dt_sl, const float *A,
                                    int64_t B, int64_t L, int64_t H, float *out, cudaStream_t s);
cudaError_t launch_sequence_combine(const float *logdecay, const float *states, const float *h0,
                                    int rank, int64_t BH, int64_t PN, float *h_in, cudaStream_t s);
cudaError_t launch_shard_correct(const Args &a, const float *h_in, const float *logdecay,
                                 cudaStream_t s);
}  // namespace ssd

ssd_status ssd_segment_logdecay(const ssd_tensor *dt, const ssd_tensor *A, ssd_tensor *logdecay,
                                void *stream) {
    if (!dt || dt->ndim != 3) return fail(SSD_ERR_INVALID_ARG, "dt: missing or ndim != 3");
    const int64_t Bn = dt->shape[0], L = dt->shape[1], H = dt->shape[2];
    if (Bn < 0 || L < 0 || H <= 0 || H > 65535 || Bn > 65535)
        return fail(SSD_ERR_INVALID_ARG, "dt: shape (%lld, %lld, %lld) out of range",
                    (long long)Bn, (long long)L, (long long)H);
    const int64_t sdt[3] = {Bn, L, H}, sh[1] = {H}, so[2] = {Bn, H};
    ssd_status st;
    if ((st = check_tensor(dt, "dt", 3, sdt, SSD_F32, false, false))) return st;
    if ((st = check_tensor(A, "A", 1, sh, SSD_F32, true, false))) return st;
    if ((st = check_tensor(logdecay, "logdecay", 2, so, SSD_F32, true, false))) return st;
    const Range ro = range_of(logdecay);
    if (overlap(ro, range_of(dt)) || overlap(ro, range_of(A)))
        return fail(SSD_ERR_INVALID_ARG, "logdecay overlaps an input");
    if (Bn == 0) return ok();
    if ((st = check_device_ptrs({{dt->data, "dt"}, {A->data, "A"}, {logdecay->data, "logdecay"}})))
        return st;
    if ((st = cuda_status(ssd::launch_segment_logdecay(
                              static_cast<const float *>(dt->data), dt->stride[0], dt->stride[1],
                              static_cast<const float *>(A->data), Bn, L, H,
                              static_cast<float *>(logdecay->data),
                              static_cast<cudaStream_t>(stream)),
                          "segment log-decay")))
        return st;
    return ok();
}

ssd_status ssd_sequence_combine(const ssd_tensor *logdecay_all, const ssd_tensor *states_all,
                                const ssd_tensor *initial_states, int32_t rank, ssd_tensor *h_in,
                                void *stream) {
    if (!states_all || states_all->ndim != 5)
        return fail(SSD_ERR_INVALID_ARG, "states: missing or ndim != 5");
    const int64_t R = states_all->shape[0], Bn = states_all->shape[1], H = states_all->shape[2],
                  P = states_all->shape[3], N = states_all->shape[4];
    if (R <= 0 || rank < 0 || rank >= R)
        return fail(SSD_ERR_INVALID_ARG, "rank %d outside [0, %lld)", rank, (long long)R);
    const int64_t sl[3] = {R, Bn, H}, ss[5] = {R, Bn, H, P, N}, sh[4] = {Bn, H, P, N};
    ssd_status st;
    if ((st = check_tensor(logdecay_all, "logdecay", 3, sl, SSD_F32, true, false))) return st;
    if ((st = check_tensor(states_all, "states", 5, ss, SSD_F32, true, false))) return st;
    if (initial_states &&
        (st = check_tensor(initial_states, "initial_states", 4, sh, SSD_F32, true, false)))
        return st;
    if ((st = check_tensor(h_in, "h_in", 4, sh, SSD_F32, true, false))) return st;
    const Range ro = range_of(h_in);
    if (overlap(ro, range_of(logdecay_all)) || overlap(ro, range_of(states_all)) ||
        overlap(ro, range_of(initial_states)))
        return fail(SSD_ERR_INVALID_ARG, "h_in overlaps an input");
    if (Bn * H * P * N == 0) return ok();
    if ((st = check_device_ptrs({{logdecay_all->data, "logdecay"}, {states_all->data, "states"},
                                 {initial_states ? initial_states->data : nullptr,
                                  "initial_states"},
                                 {h_in->data, "h_in"}})))
        return st;
    if ((st = cuda_status(ssd::launch_sequence_combine(
                              static_cast<const float *>(logdecay_all->data),
                              static_cast<const float *>(states_all->data),
                              initial_states ? static_cast<const float *>(initial_states->data)
                                             : nullptr,
                              rank, Bn * H, P * N, static_cast<float *>(h_in->data),
                              static_cast<cudaStream_t>(stream)),
                          "sequence combine")))
        return st;
    return ok();
}

ssd_status ssd_shard_correct(const ssd_tensor *dt, const ssd_tensor *A, const ssd_tensor *Cm,
                             const ssd_tensor *h_in, const ssd_tensor *logdecay, int64_t ngroups,
                             ssd_tensor *y, ssd_tensor *final_states, void *stream) {
    if (!y || !Cm) return fail(SSD_ERR_INVALID_ARG, "y / C: null tensor descriptor");
    if (y->ndim != 4 || Cm->ndim != 4) return fail(SSD_ERR_INVALID_ARG, "y / C: ndim must be 4");
    const int64_t Bn = y->shape[0], L = y->shape[1], H = y->shape[2], P = y->shape[3];
    const int64_t N = Cm->shape[3], Gn = ngroups;
    ssd_status st = check_geometry(Bn, L, H, P, N, Gn, 256);
    if (st != SSD_OK) return st;
    const int xdt = y->dtype;
    const int64_t sy[4] = {Bn, L, H, P}, sdt[3] = {Bn, L, H}, sc[4] = {Bn, L, Gn, N},
                  sh[1] = {H}, sst[4] = {Bn, H, P, N}, sld[2] = {Bn, H};
    if ((st = check_tensor(y, "y", 4, sy, -1, false, false))) return st;
    if ((st = check_tensor(dt, "dt", 3, sdt, SSD_F32, false, false))) return st;
    if ((st = check_tensor(A, "A", 1, sh, SSD_F32, true, false))) return st;
    if ((st = check_tensor(Cm, "C", 4, sc, xdt, false, false))) return st;
    if ((st = check_tensor(h_in, "h_in", 4, sst, SSD_F32, true, false))) return st;
    if ((st = check_tensor(logdecay, "logdecay", 2, sld, SSD_F32, true, false))) return st;
    if (final_states &&
        (st = check_tensor(final_states, "final_states", 4, sst, SSD_F32, true, false)))
        return st;
    const Range ry = range_of(y), rf = range_of(final_states);
    const Range ins[] = {range_of(dt), range_of(A), range_of(Cm), range_of(h_in),
                         range_of(logdecay)};
    for (const Range &r : ins)
        if (overlap(ry, r) || overlap(rf, r))
            return fail(SSD_ERR_INVALID_ARG, "an output overlaps an input");
    if (overlap(ry, rf)) return fail(SSD_ERR_INVALID_ARG, "y overlaps final_states");
    if (Bn == 0) return ok();
    if ((st = check_device_ptrs({{dt->data, "dt"}, {A->data, "A"}, {Cm->data, "C"},
                                 {h_in->data, "h_in"}, {logdecay->data, "logdecay"},
                                 {y->data, "y"},
                                 {final_states ? final_states->data : nullptr, "final_states"}})))
        return st;
    ssd::Args a;
    a.d = ssd::Dims{Bn, L, H, P, N, Gn, 256, (L + 255) / 256};
    a.xdt = xdt;
    fill_dt(a, dt);
    a.A = static_cast<const float *>(A->data);
    fill_bc(a, nullptr, Cm);
    fill_y(a, y);
    a.final_states = final_states ? static_cast<float *>(final_states->data) : nullptr;
    if ((st = cuda_status(ssd::launch_shard_correct(a, static_cast<const float *>(h_in->data),
                                                    static_cast<const float *>(logdecay->data),
                                                    static_cast<cudaStream_t>(stream)),
                          "shard correction")))
        return st;
    return ok();
}
