// C ABI of libhg.so: argument checking, the level schedule, per-level
// constants, layout detection, and dispatch to the kernels.  Declared in
// include/hg.h, which also documents every entry point.
#include <cuda_runtime.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <cmath>
#include <cstdint>

#include "hg_params.h"
#include "../../include/hg_probe.h"

namespace {

thread_local char g_err[512] = "";

hg_status fail(hg_status s, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return s;
}

hg_status ok() {
    g_err[0] = '\0';
    return HG_OK;
}

int binom(int n, int k) {
    int r = 1;
    for (int i = 0; i < k; ++i) r = r * (n - i) / (i + 1);
    return r;
}

// ---------------------------------------------------------------------------
// Level schedule: N_l = floor(n_min * (n_max/n_min)^(l/(L-1))).  A double
// estimate is corrected with an exact integer test
//     n^(L-1) <= n_max^l * n_min^(L-1-l)
// evaluated on little-endian base-2^32 big integers.
// ---------------------------------------------------------------------------
struct Big {
    uint32_t w[48];
    int n;
};

void big_set(Big& b, uint32_t v) {
    b.w[0] = v;
    b.n = 1;
}

void big_mul(Big& b, uint32_t m) {
    uint64_t carry = 0;
    for (int i = 0; i < b.n; ++i) {
        const uint64_t cur = static_cast<uint64_t>(b.w[i]) * m + carry;
        b.w[i] = static_cast<uint32_t>(cur);
        carry = cur >> 32;
    }
    if (carry) b.w[b.n++] = static_cast<uint32_t>(carry);
    while (b.n > 1 && b.w[b.n - 1] == 0) --b.n;
}

int big_cmp(const Big& a, const Big& b) {
    if (a.n != b.n) return a.n < b.n ? -1 : 1;
    for (int i = a.n - 1; i >= 0; --i)
        if (a.w[i] != b.w[i]) return a.w[i] < b.w[i] ? -1 : 1;
    return 0;
}

// n^(L-1) <= n_max^l * n_min^(L-1-l)
bool at_most_exact(uint32_t n, int L, int l, uint32_t n_min, uint32_t n_max) {
    Big lhs, rhs;
    big_set(lhs, 1);
    big_set(rhs, 1);
    for (int i = 0; i < L - 1; ++i) big_mul(lhs, n);
    for (int i = 0; i < l; ++i) big_mul(rhs, n_max);
    for (int i = 0; i < L - 1 - l; ++i) big_mul(rhs, n_min);
    return big_cmp(lhs, rhs) <= 0;
}

hg_status compute_resolutions(const hg_grid_desc* desc, int32_t* res) {
    const int L = desc->L;
    if (desc->res) {
        for (int l = 0; l < L; ++l) {
            if (desc->res[l] < 1 || desc->res[l] > HG_MAX_RESOLUTION)
                return fail(HG_ERR_INVALID_ARG, "res[%d] = %d is outside 1..%d", l, desc->res[l], HG_MAX_RESOLUTION);
            res[l] = desc->res[l];
        }
        return HG_OK;
    }
    const int64_t n_min = desc->n_min, n_max = desc->n_max;
    if (n_min < 1 || n_max < n_min || n_max > HG_MAX_RESOLUTION)
        return fail(HG_ERR_INVALID_ARG, "need 1 <= n_min (%lld) <= n_max (%lld) <= %d", (long long)n_min,
                    (long long)n_max, HG_MAX_RESOLUTION);
    if (L == 1) {
        res[0] = static_cast<int32_t>(n_min);
        return HG_OK;
    }
    const double lb = std::log(static_cast<double>(n_max) / static_cast<double>(n_min)) / (L - 1);
    for (int l = 0; l < L; ++l) {
        int64_t est = static_cast<int64_t>(std::floor(static_cast<double>(n_min) * std::exp(lb * l)));
        est = est < n_min ? n_min : (est > n_max ? n_max : est);
        while (est > n_min && !at_most_exact(static_cast<uint32_t>(est), L, l, n_min, n_max)) --est;
        while (est < n_max && at_most_exact(static_cast<uint32_t>(est + 1), L, l, n_min, n_max)) ++est;
        res[l] = static_cast<int32_t>(est);
    }
    return HG_OK;
}

// ---------------------------------------------------------------------------
// common checks and parameter blocks
// ---------------------------------------------------------------------------
size_t dtype_size(int dtype) { return dtype == HG_F16 ? 2 : 4; }

hg_status check_desc(const hg_grid_desc* desc, int n_orders) {
    if (!desc) return fail(HG_ERR_INVALID_ARG, "desc is NULL");
    if (desc->d < 2 || desc->d > 4) return fail(HG_ERR_INVALID_ARG, "d = %d; must be 2, 3 or 4", desc->d);
    if (desc->L < 1 || desc->L > HG_MAX_LEVELS)
        return fail(HG_ERR_INVALID_ARG, "L = %d; must be in 1..%d", desc->L, HG_MAX_LEVELS);
    if (desc->F != 1 && desc->F != 2 && desc->F != 4 && desc->F != 8)
        return fail(HG_ERR_INVALID_ARG, "F = %d; must be 1, 2, 4 or 8", desc->F);
    if (desc->dtype != HG_F32 && desc->dtype != HG_F16) return fail(HG_ERR_INVALID_ARG, "unknown dtype %d", desc->dtype);
    if (desc->layout != HG_POINT_MAJOR && desc->layout != HG_FEATURE_MAJOR)
        return fail(HG_ERR_INVALID_ARG, "unknown layout %d", desc->layout);
    for (int k = 0; k < n_orders; ++k)
        if (desc->log2_T[k] < 0 || desc->log2_T[k] > HG_MAX_LOG2_T)
            return fail(HG_ERR_INVALID_ARG, "log2_T[%d] = %d; must be in 0..%d", k, desc->log2_T[k], HG_MAX_LOG2_T);
    if (desc->L < 32 && (desc->level_mask >> desc->L) != 0)
        return fail(HG_ERR_INVALID_ARG, "level_mask 0x%x has bits at or above L = %d", desc->level_mask, desc->L);
    return HG_OK;
}

hg_status check_n(int64_t n) {
    if (n < 0 || n > INT32_MAX) return fail(HG_ERR_INVALID_ARG, "n = %lld; must be in 0..2^31-1", (long long)n);
    return HG_OK;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Fills c from desc (orders 0..n_orders-1 decide the dense flags).
hg_status make_common(const hg_grid_desc* desc, int n_orders, int64_t n, hg::Common& c) {
    memset(&c, 0, sizeof(c));
    c.d = desc->d;
    c.L = desc->L;
    c.F = desc->F;
    c.level_mask = desc->level_mask;
    c.n = n;
    int32_t res[HG_MAX_LEVELS];
    hg_status st = compute_resolutions(desc, res);
    if (st != HG_OK) return st;
    for (int k = 0; k < 5; ++k) c.tmask[k] = k < n_orders ? (1u << desc->log2_T[k]) - 1u : 0u;
    for (int l = 0; l < desc->L; ++l) {
        hg::Level& lv = c.lv[l];
        const uint32_t N = static_cast<uint32_t>(res[l]);
        lv.N = N;
        lv.side = N + 1;
        lv.side2 = (N + 1) * (N + 1);  // only used when the level is one-to-one (fits 2^30)
        lv.side3 = static_cast<uint32_t>(static_cast<uint64_t>(N + 1) * (N + 1) * (N + 1));  // likewise (4D)
        lv.fN = static_cast<float>(N);
        lv.fN2 = static_cast<float>(static_cast<double>(N) * N);
        lv.dx = static_cast<float>(1.0 / N);
        lv.dense = 0;
        for (int k = 0; k < n_orders; ++k) {
            const uint64_t T = uint64_t(1) << desc->log2_T[k];
            uint64_t verts = 1;
            bool fits = true;
            for (int i = 0; i < desc->d; ++i) {
                verts *= (uint64_t)N + 1;
                if (verts > T) {
                    fits = false;
                    break;
                }
            }
            if (fits) lv.dense |= 1u << k;
        }
    }
    const int64_t LF = static_cast<int64_t>(desc->L) * desc->F;
    const int P = desc->d * (desc->d + 1) / 2;  // Hessian entries (upper triangle)
    if (desc->layout == HG_POINT_MAJOR) {
        c.sn = LF;
        c.sf = 1;
        c.dsn = desc->d * LF;
        c.dsj = LF;
        c.dsf = 1;
        c.hsn = P * LF;
        c.hsq = LF;
        c.hsf = 1;
        c.ssn = 2 * desc->d * LF;
        c.ssj = LF;
        c.ssf = 1;
    } else {
        c.sn = 1;
        c.sf = n;
        c.dsn = 1;
        c.dsj = LF * n;
        c.dsf = n;
        c.hsn = 1;
        c.hsq = LF * n;
        c.hsf = n;
        c.ssn = 1;
        c.ssj = LF * n;
        c.ssf = n;
    }
    return HG_OK;
}

// A table view: non-NULL, element-aligned, rows that do not overlap.
hg_status check_view(const char* what, int k, const void* ptr, int64_t ls, int64_t rs, int64_t width, int64_t T,
                     int L, size_t esize) {
    if (!ptr) return fail(HG_ERR_INVALID_ARG, "%s[%d].ptr is NULL", what, k);
    if (!aligned(ptr, esize)) return fail(HG_ERR_INVALID_ARG, "%s[%d].ptr is not %zu-byte aligned", what, k, esize);
    if (rs < width)
        return fail(HG_ERR_INVALID_ARG, "%s[%d].row_stride = %lld < %lld values per entry", what, k, (long long)rs,
                    (long long)width);
    if (L > 1 && ls < T * rs)
        return fail(HG_ERR_INVALID_ARG, "%s[%d].level_stride = %lld < T * row_stride = %lld", what, k, (long long)ls,
                    (long long)(T * rs));
    if (ls < 0) return fail(HG_ERR_INVALID_ARG, "%s[%d].level_stride is negative", what, k);
    return HG_OK;
}

// True when the d+1 views are the interleaved [L][T][2^d][F] buffer.
bool is_packed(const hg_grid_desc* desc, const void* const* ptrs, const int64_t* ls, const int64_t* rs, size_t esize) {
    const int d = desc->d, F = desc->F, V = 1 << d;
    int off = 0;
    for (int k = 0; k <= d; ++k) {
        if (desc->log2_T[k] != desc->log2_T[0]) return false;
        if (rs[k] != static_cast<int64_t>(V) * F || ls[k] != ls[0]) return false;
        const char* want = static_cast<const char*>(ptrs[0]) + static_cast<size_t>(off) * F * esize;
        if (static_cast<const char*>(ptrs[k]) != want) return false;
        off += binom(d, k);
    }
    return true;
}

// Launches cover every level (the forwards write zeros for inactive ones).
void all_levels(hg::Common& c) {
    c.nlvl = c.L;
    for (int l = 0; l < c.L; ++l) c.lvl[l] = static_cast<uint8_t>(l);
}

// Streaming multiprocessors of the current device (148 if it cannot be read).
int sm_count() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && sms > 0)
        return sms;
    return 148;
}

// Shared memory per CTA of the privatised backward, and the largest whole
// level (all parts of its rows) the Hermite backward privatises.  Measured on
// B300: a d-linear level of up to ~100 KB gains several times over direct
// REDs (a few hundred hot rows serialise in L2), while Hermite levels gain
// only when tiny -- 3D levels of hundreds of KB run at the full RED rate
// directly, and the shared-memory pass then costs more than it saves.  2D
// PINN grid (2^20 points, one level per launch): the 289- and 484-row levels
// (9 and 15 KB) take 0.12 ms privatised against 0.18 ms direct when the
// points come in random order, but the 784-row level (25 KB) 0.12 against
// 0.08 ms; points in stratum order sum their runs in the warp and run faster
// direct at every level (whole backward 0.66 ms privatising up to 32 KB,
// 0.56 ms direct).
constexpr int64_t kPrivMaxBytes = 160 * 1024;
constexpr int64_t kHermitePrivLevelBytes = 16 * 1024;

// Splits the active levels of a backward between the privatised kernel
// (one-to-one levels whose rows -- part_bytes per row and CTA -- fit in
// shared memory, whose whole size is at most level_limit, and which receive
// many contributions per row) and the direct kernel.  parts = CTAs sharing a
// row (16-byte parts of a Hermite row).
void plan_backward(hg::BwdParams& p, bool allow, int64_t part_bytes, int parts, int64_t level_limit) {
    hg::Common& c = p.c;
    const int V = 1 << c.d;
    const int64_t target = 2 * static_cast<int64_t>(sm_count());
    bool cand[HG_MAX_LEVELS] = {};
    uint64_t rows[HG_MAX_LEVELS] = {};
    int ncand = 0;
    for (int l = 0; l < c.L; ++l) {
        if (!((c.level_mask >> l) & 1u) || !allow || !(c.lv[l].dense & 1u)) continue;
        rows[l] = 1;
        for (int i = 0; i < c.d; ++i) rows[l] *= c.lv[l].side;
        if (static_cast<int64_t>(rows[l]) * part_bytes <= kPrivMaxBytes &&
            static_cast<int64_t>(rows[l]) * part_bytes * parts <= level_limit) {
            cand[l] = true;
            ++ncand;
        }
    }
    // each privatised CTA flushes all its rows: keep a level only if its
    // contributions outnumber the flushed rows severalfold
    int64_t chunks = 1;
    for (int pass = 0; pass < 2 && ncand > 0; ++pass) {
        chunks = (target + static_cast<int64_t>(ncand) * parts - 1) / (static_cast<int64_t>(ncand) * parts);
        if (chunks < 1) chunks = 1;
        ncand = 0;
        for (int l = 0; l < c.L; ++l) {
            if (!cand[l]) continue;
            if (c.n * V < 4 * static_cast<int64_t>(rows[l]) * chunks) cand[l] = false;
            else ++ncand;
        }
    }
    c.nlvl = 0;
    p.priv.n = 0;
    p.priv.smem_bytes = 0;
    for (int l = 0; l < c.L; ++l) {
        if (!((c.level_mask >> l) & 1u)) continue;
        if (cand[l]) {
            p.priv.lvl[p.priv.n] = static_cast<uint8_t>(l);
            p.priv.rows[p.priv.n] = static_cast<uint32_t>(rows[l]);
            const int64_t b = static_cast<int64_t>(rows[l]) * part_bytes;
            if (b > p.priv.smem_bytes) p.priv.smem_bytes = static_cast<int32_t>(b);
            ++p.priv.n;
        } else {
            c.lvl[c.nlvl++] = static_cast<uint8_t>(l);
        }
    }
    p.priv.chunk = (c.n + chunks - 1) / chunks;
    if (p.priv.chunk < 1) p.priv.chunk = 1;
}

hg_status launch_status(int err, const char* what) {
    if (err != cudaSuccess)
        return fail(HG_ERR_CUDA, "%s launch failed: %s", what, cudaGetErrorString(static_cast<cudaError_t>(err)));
    return ok();
}

// Hermite forward, Laplacian or (hess) full-Hessian outputs in `second`.
hg_status hermite_forward(const hg_grid_desc* desc, int64_t n, const float* coords, const hg_table* tables,
                          float* gamma, float* dgamma, float* second, bool hess, hg_stream stream) {
    hg_status st = check_desc(desc, desc ? desc->d + 1 : 0);
    if (st != HG_OK) return st;
    if ((st = check_n(n)) != HG_OK) return st;
    if (!tables) return fail(HG_ERR_INVALID_ARG, "tables is NULL");
    const int d = desc->d, F = desc->F, V = 1 << d;
    const size_t es = dtype_size(desc->dtype);
    const void* ptrs[5];
    int64_t ls[5], rs[5];
    for (int k = 0; k <= d; ++k) {
        ptrs[k] = tables[k].ptr;
        ls[k] = tables[k].level_stride;
        rs[k] = tables[k].row_stride;
        st = check_view("tables", k, ptrs[k], ls[k], rs[k], static_cast<int64_t>(binom(d, k)) * F,
                        int64_t(1) << desc->log2_T[k], desc->L, es);
        if (st != HG_OK) return st;
    }
    hg::FwdParams p;
    if ((st = make_common(desc, d + 1, n, p.c)) != HG_OK) return st;
    if (n == 0) return ok();
    if (!coords || !gamma) return fail(HG_ERR_INVALID_ARG, "coords and gamma must not be NULL");
    if (hess && !second) return fail(HG_ERR_INVALID_ARG, "hess must not be NULL");
    if (!aligned(coords, 4) || !aligned(gamma, 4) || (dgamma && !aligned(dgamma, 4)) ||
        (second && !aligned(second, 4)))
        return fail(HG_ERR_INVALID_ARG, "coords and outputs must be 4-byte aligned");
    for (int k = 0; k <= d; ++k) {
        p.tab.ptr[k] = ptrs[k];
        p.tab.ls[k] = ls[k];
        p.tab.rs[k] = rs[k];
    }
    p.coords = coords;
    p.gamma = gamma;
    p.dgamma = dgamma;
    p.lap = hess ? nullptr : second;
    p.hess = hess ? second : nullptr;
    p.stencil = nullptr;
    const int fc = (F % 2 == 0) ? 2 : 1;
    bool vec = fc == F && is_packed(desc, ptrs, ls, rs, es);
    if (vec) {
        const size_t row = static_cast<size_t>(V) * F * es;
        const size_t al = row < 32 ? row : 32;  // 256-bit loads of 32-byte rows / half-rows
        vec = aligned(ptrs[0], al) && (static_cast<size_t>(ls[0]) * es) % al == 0;
    }
    all_levels(p.c);
    return launch_status(hg::launch_hermite_fwd(p, fc, vec, desc->dtype, hess, stream),
                         hess ? "hermite forward (Hessian)" : "hermite forward");
}

// Hermite backward, upstream gradient of the Laplacian or (hess) of the
// full Hessian in `g_second`.
hg_status hermite_backward(const hg_grid_desc* desc, int64_t n, const float* coords, const float* g_gamma,
                           const float* g_dgamma, const float* g_second, const hg_grad_table* grads, bool hess,
                           hg_stream stream) {
    hg_status st = check_desc(desc, desc ? desc->d + 1 : 0);
    if (st != HG_OK) return st;
    if ((st = check_n(n)) != HG_OK) return st;
    if (!grads) return fail(HG_ERR_INVALID_ARG, "grads is NULL");
    const int d = desc->d, F = desc->F, V = 1 << d;
    const void* ptrs[5];
    int64_t ls[5], rs[5];
    for (int k = 0; k <= d; ++k) {
        ptrs[k] = grads[k].ptr;
        ls[k] = grads[k].level_stride;
        rs[k] = grads[k].row_stride;
        st = check_view("grads", k, ptrs[k], ls[k], rs[k], static_cast<int64_t>(binom(d, k)) * F,
                        int64_t(1) << desc->log2_T[k], desc->L, 4);
        if (st != HG_OK) return st;
    }
    hg::BwdParams p;
    if ((st = make_common(desc, d + 1, n, p.c)) != HG_OK) return st;
    if (n == 0 || (!g_gamma && !g_dgamma && !g_second)) return ok();
    if (!coords) return fail(HG_ERR_INVALID_ARG, "coords must not be NULL");
    if (!aligned(coords, 4) || (g_gamma && !aligned(g_gamma, 4)) || (g_dgamma && !aligned(g_dgamma, 4)) ||
        (g_second && !aligned(g_second, 4)))
        return fail(HG_ERR_INVALID_ARG, "coords and upstream gradients must be 4-byte aligned");
    for (int k = 0; k <= d; ++k) {
        p.grad.ptr[k] = const_cast<float*>(static_cast<const float*>(ptrs[k]));
        p.grad.ls[k] = ls[k];
        p.grad.rs[k] = rs[k];
    }
    p.coords = coords;
    p.g_gamma = g_gamma;
    p.g_dgamma = g_dgamma;
    p.g_lap = hess ? nullptr : g_second;
    p.g_hess = hess ? g_second : nullptr;
    p.g_stencil = nullptr;
    const int fc = (F % 2 == 0) ? 2 : 1;
    bool vec = fc == F && is_packed(desc, ptrs, ls, rs, 4);
    if (vec) vec = aligned(ptrs[0], 16) && (static_cast<size_t>(ls[0]) * 4) % 16 == 0 && (V * F) % 4 == 0;
    // the 4D kernels scatter every level directly (no privatised variant)
    plan_backward(p, vec && d != 4, 16, vec ? V * F / 4 : 1, kHermitePrivLevelBytes);
    return launch_status(hg::launch_hermite_bwd(p, fc, vec, hess, stream),
                         hess ? "hermite backward (Hessian)" : "hermite backward");
}

// Replay probe: shared checks, parameter block and launch.
hg_status replay(const hg_grid_desc* desc, int64_t n, const float* coords, void* buf, int64_t level_bytes,
                 int32_t row_bytes, int32_t lanes, float* sink, bool red, hg_stream stream) {
    hg_status st = check_desc(desc, 1);
    if (st != HG_OK) return st;
    if ((st = check_n(n)) != HG_OK) return st;
    if (lanes < 1 || row_bytes < 4 || row_bytes % lanes != 0)
        return fail(HG_ERR_INVALID_ARG, "row_bytes %d, lanes_per_row %d: need a positive multiple", row_bytes, lanes);
    const int ch = row_bytes / lanes;
    if (!(ch == 4 || ch == 8 || ch == 16 || (ch == 32 && !red)))
        return fail(HG_ERR_INVALID_ARG, "unsupported chunk of %d bytes", ch);
    const int64_t T = int64_t(1) << desc->log2_T[0];
    if (desc->L > 1 && level_bytes < T * row_bytes)
        return fail(HG_ERR_INVALID_ARG, "level_stride_bytes %lld < T * row_bytes", (long long)level_bytes);
    if (level_bytes < 0 || level_bytes % ch != 0 || row_bytes % ch != 0)
        return fail(HG_ERR_INVALID_ARG, "strides must be non-negative multiples of the %d-byte chunk", ch);
    hg::ReplayParams p;
    if ((st = make_common(desc, 1, n, p.c)) != HG_OK) return st;
    if (n == 0) return ok();
    if (!coords || !buf || (!red && !sink)) return fail(HG_ERR_INVALID_ARG, "NULL coords, table or sink");
    if (!aligned(coords, 4) || !aligned(buf, ch) || (sink && !aligned(sink, 4)))
        return fail(HG_ERR_INVALID_ARG, "coords / sink must be 4-byte and the table chunk-aligned");
    all_levels(p.c);
    p.coords = coords;
    p.base = static_cast<char*>(buf);
    p.level_bytes = level_bytes;
    p.row_bytes = row_bytes;
    p.lanes = lanes;
    p.sink = sink;
    return launch_status(hg::launch_replay(p, red, stream), "replay probe");
}

// Finite-difference step checks and the fp32 factors 1/(2 eps), 1/eps^2.
hg_status fd_step(float eps, float& half_inv, float& inv2) {
    if (!(eps > 0.0f) || !(eps < INFINITY)) return fail(HG_ERR_INVALID_ARG, "eps = %g; must be positive and finite", eps);
    const double e = eps;
    half_inv = static_cast<float>(1.0 / (2.0 * e));
    inv2 = static_cast<float>(1.0 / (e * e));
    if (!(inv2 < INFINITY)) return fail(HG_ERR_INVALID_ARG, "eps = %g is too small (1/eps^2 overflows)", eps);
    return HG_OK;
}


// SIREN consumer: argument checks and the tile plan (threads per point, points per tile,
// weight-gradient splits), then one wave of persistent CTAs.
hg_status siren_plan(const hg_siren_desc* desc, int64_t n, hg::SirenParams& p) {
    if (!desc) return fail(HG_ERR_INVALID_ARG, "desc is NULL");
    hg_status st = check_n(n);
    if (st != HG_OK) return st;
    if (desc->d < 1 || desc->d > 4) return fail(HG_ERR_INVALID_ARG, "d = %d; must be in 1..4", desc->d);
    if (desc->K < 8 || desc->K > 64 || desc->K % 8 != 0)
        return fail(HG_ERR_INVALID_ARG, "K = %d; must be a multiple of 8 in 8..64", desc->K);
    if (desc->H != 16 && desc->H != 32 && desc->H != 64 && desc->H != 128)
        return fail(HG_ERR_INVALID_ARG, "H = %d; must be 16, 32, 64 or 128", desc->H);
    if (desc->O < 1 || desc->O > 4) return fail(HG_ERR_INVALID_ARG, "O = %d; must be in 1..4", desc->O);
    if (!(fabsf(desc->omega) < INFINITY)) return fail(HG_ERR_INVALID_ARG, "omega must be finite");
    memset(&p, 0, sizeof(p));
    p.d = desc->d;
    p.K = desc->K;
    p.H = desc->H;
    p.O = desc->O;
    p.tp = desc->H / 16;
    p.nbuf = 1;
    p.pts = 256 / p.tp;
    p.n = n;
    p.omega = desc->omega;
    return HG_OK;
}

// Largest opt-in shared memory per block of the current device.
hg_status query_smem_max(int& smem_max) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&smem_max, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    return e == cudaSuccess ? HG_OK : HG_ERR_CUDA;
}

// One wave of persistent CTAs for a planned launch (n > 0), and the number of input buffers.
hg_status siren_grid(hg::SirenParams& p, bool bwd, int& ctas) {
    const int64_t n = p.n;
    int dev = 0, sms = 0, smem_max = 0, per_sm = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&smem_max, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) return fail(HG_ERR_CUDA, "device query failed: %s", cudaGetErrorString(e));
    // two input buffers (the next tile's copy overlapping this one's compute) when they fit
    p.nbuf = 2;
    if (hg::siren_smem_bytes(p, bwd) > static_cast<size_t>(smem_max)) p.nbuf = 1;
    const size_t bytes = hg::siren_smem_bytes(p, bwd);
    if (bytes > static_cast<size_t>(smem_max))
        return fail(HG_ERR_UNSUPPORTED, "a SIREN tile needs %zu bytes of shared memory (at most %d)", bytes, smem_max);
    e = static_cast<cudaError_t>(hg::siren_ctas_per_sm(p, bwd, &per_sm));
    if (e != cudaSuccess || per_sm < 1) return fail(HG_ERR_CUDA, "SIREN occupancy query failed");
    const int64_t tiles = (n + p.pts - 1) / p.pts;
    ctas = static_cast<int>(std::min<int64_t>(tiles, static_cast<int64_t>(sms) * per_sm));
    return HG_OK;
}

}  // namespace

extern "C" {

int32_t hg_abi_version(void) { return HG_ABI_VERSION; }

const char* hg_status_string(hg_status s) {
    switch (s) {
        case HG_OK: return "HG_OK";
        case HG_ERR_INVALID_ARG: return "HG_ERR_INVALID_ARG";
        case HG_ERR_UNSUPPORTED: return "HG_ERR_UNSUPPORTED";
        case HG_ERR_CUDA: return "HG_ERR_CUDA";
    }
    return "HG_UNKNOWN_STATUS";
}

const char* hg_last_error(void) { return g_err; }

hg_status hg_level_resolutions(const hg_grid_desc* desc, int32_t* res_out) {
    if (!desc) return fail(HG_ERR_INVALID_ARG, "desc is NULL");
    if (!res_out) return fail(HG_ERR_INVALID_ARG, "res_out is NULL");
    if (desc->L < 1 || desc->L > HG_MAX_LEVELS)
        return fail(HG_ERR_INVALID_ARG, "L = %d; must be in 1..%d", desc->L, HG_MAX_LEVELS);
    hg_status st = compute_resolutions(desc, res_out);
    return st == HG_OK ? ok() : st;
}

hg_status hg_encode_fwd(const hg_grid_desc* desc, int64_t n, const float* coords, const hg_table* tables,
                        float* gamma, float* dgamma, float* lap, hg_stream stream) {
    return hermite_forward(desc, n, coords, tables, gamma, dgamma, lap, false, stream);
}

hg_status hg_encode_fwd_hessian(const hg_grid_desc* desc, int64_t n, const float* coords, const hg_table* tables,
                                float* gamma, float* dgamma, float* hess, hg_stream stream) {
    return hermite_forward(desc, n, coords, tables, gamma, dgamma, hess, true, stream);
}

hg_status hg_encode_bwd(const hg_grid_desc* desc, int64_t n, const float* coords, const float* g_gamma,
                        const float* g_dgamma, const float* g_lap, const hg_grad_table* grads, hg_stream stream) {
    return hermite_backward(desc, n, coords, g_gamma, g_dgamma, g_lap, grads, false, stream);
}

hg_status hg_encode_bwd_hessian(const hg_grid_desc* desc, int64_t n, const float* coords, const float* g_gamma,
                                const float* g_dgamma, const float* g_hess, const hg_grad_table* grads,
                                hg_stream stream) {
    return hermite_backward(desc, n, coords, g_gamma, g_dgamma, g_hess, grads, true, stream);
}

hg_status hg_linear_fwd(const hg_grid_desc* desc, int64_t n, const float* coords, const hg_table* table,
                        float* gamma, hg_stream stream) {
    hg_status st = check_desc(desc, 1);
    if (st != HG_OK) return st;
    if ((st = check_n(n)) != HG_OK) return st;
    if (!table) return fail(HG_ERR_INVALID_ARG, "table is NULL");
    const int F = desc->F;
    const size_t es = dtype_size(desc->dtype);
    st = check_view("table", 0, table->ptr, table->level_stride, table->row_stride, F, int64_t(1) << desc->log2_T[0],
                    desc->L, es);
    if (st != HG_OK) return st;
    hg::FwdParams p;
    if ((st = make_common(desc, 1, n, p.c)) != HG_OK) return st;
    if (n == 0) return ok();
    if (!coords || !gamma) return fail(HG_ERR_INVALID_ARG, "coords and gamma must not be NULL");
    if (!aligned(coords, 4) || !aligned(gamma, 4)) return fail(HG_ERR_INVALID_ARG, "coords and gamma must be 4-byte aligned");
    memset(&p.tab, 0, sizeof(p.tab));
    p.tab.ptr[0] = table->ptr;
    p.tab.ls[0] = table->level_stride;
    p.tab.rs[0] = table->row_stride;
    p.coords = coords;
    p.gamma = gamma;
    p.dgamma = nullptr;
    p.lap = nullptr;
    p.hess = nullptr;
    p.stencil = nullptr;
    const int fc = (F % 2 == 0) ? 2 : 1;
    const bool vec = fc == 2 && aligned(table->ptr, 2 * es) && table->row_stride % 2 == 0 && table->level_stride % 2 == 0;
    all_levels(p.c);
    return launch_status(hg::launch_linear_fwd(p, fc, vec, desc->dtype, stream), "linear forward");
}

hg_status hg_linear_bwd(const hg_grid_desc* desc, int64_t n, const float* coords, const float* g_gamma,
                        const hg_grad_table* grad, hg_stream stream) {
    hg_status st = check_desc(desc, 1);
    if (st != HG_OK) return st;
    if ((st = check_n(n)) != HG_OK) return st;
    if (!grad) return fail(HG_ERR_INVALID_ARG, "grad is NULL");
    const int F = desc->F;
    st = check_view("grad", 0, grad->ptr, grad->level_stride, grad->row_stride, F, int64_t(1) << desc->log2_T[0],
                    desc->L, 4);
    if (st != HG_OK) return st;
    hg::BwdParams p;
    if ((st = make_common(desc, 1, n, p.c)) != HG_OK) return st;
    if (n == 0 || !g_gamma) return ok();
    if (!coords) return fail(HG_ERR_INVALID_ARG, "coords must not be NULL");
    if (!aligned(coords, 4) || !aligned(g_gamma, 4))
        return fail(HG_ERR_INVALID_ARG, "coords and g_gamma must be 4-byte aligned");
    memset(&p.grad, 0, sizeof(p.grad));
    p.grad.ptr[0] = grad->ptr;
    p.grad.ls[0] = grad->level_stride;
    p.grad.rs[0] = grad->row_stride;
    p.coords = coords;
    p.g_gamma = g_gamma;
    p.g_dgamma = nullptr;
    p.g_lap = nullptr;
    p.g_hess = nullptr;
    p.g_stencil = nullptr;
    const int fc = (F % 2 == 0) ? 2 : 1;
    const bool vec = fc == 2 && aligned(grad->ptr, 8) && grad->row_stride % 2 == 0 && grad->level_stride % 2 == 0;
    plan_backward(p, true, static_cast<int64_t>(F) * 4, 1, kPrivMaxBytes);
    return launch_status(hg::launch_linear_bwd(p, fc, vec, stream), "linear backward");
}

hg_status hg_linear_fd_fwd(const hg_grid_desc* desc, int64_t n, const float* coords, float eps, const hg_table* table,
                           float* gamma, float* dgamma, float* lap, float* stencil, hg_stream stream) {
    hg_status st = check_desc(desc, 1);
    if (st != HG_OK) return st;
    if ((st = check_n(n)) != HG_OK) return st;
    if (!table) return fail(HG_ERR_INVALID_ARG, "table is NULL");
    hg::FwdParams p;
    if ((st = fd_step(eps, p.half_inv_eps, p.inv_eps2)) != HG_OK) return st;
    const int F = desc->F;
    const size_t es = dtype_size(desc->dtype);
    st = check_view("table", 0, table->ptr, table->level_stride, table->row_stride, F, int64_t(1) << desc->log2_T[0],
                    desc->L, es);
    if (st != HG_OK) return st;
    if ((st = make_common(desc, 1, n, p.c)) != HG_OK) return st;
    if (n == 0) return ok();
    if (!coords || !gamma) return fail(HG_ERR_INVALID_ARG, "coords and gamma must not be NULL");
    if (!aligned(coords, 4) || !aligned(gamma, 4) || (dgamma && !aligned(dgamma, 4)) || (lap && !aligned(lap, 4)) ||
        (stencil && !aligned(stencil, 4)))
        return fail(HG_ERR_INVALID_ARG, "coords and outputs must be 4-byte aligned");
    memset(&p.tab, 0, sizeof(p.tab));
    p.tab.ptr[0] = table->ptr;
    p.tab.ls[0] = table->level_stride;
    p.tab.rs[0] = table->row_stride;
    p.coords = coords;
    p.gamma = gamma;
    p.dgamma = dgamma;
    p.lap = lap;
    p.hess = nullptr;
    p.stencil = stencil;
    p.eps = eps;
    const int fc = (F % 2 == 0) ? 2 : 1;
    const bool vec = fc == 2 && aligned(table->ptr, 2 * es) && table->row_stride % 2 == 0 && table->level_stride % 2 == 0;
    all_levels(p.c);
    return launch_status(hg::launch_linear_fd_fwd(p, fc, vec, desc->dtype, stream), "finite-difference forward");
}

hg_status hg_linear_fd_bwd(const hg_grid_desc* desc, int64_t n, const float* coords, float eps, const float* g_gamma,
                           const float* g_dgamma, const float* g_lap, const float* g_stencil, const hg_grad_table* grad,
                           hg_stream stream) {
    hg_status st = check_desc(desc, 1);
    if (st != HG_OK) return st;
    if ((st = check_n(n)) != HG_OK) return st;
    if (!grad) return fail(HG_ERR_INVALID_ARG, "grad is NULL");
    hg::BwdParams p;
    if ((st = fd_step(eps, p.half_inv_eps, p.inv_eps2)) != HG_OK) return st;
    const int F = desc->F;
    st = check_view("grad", 0, grad->ptr, grad->level_stride, grad->row_stride, F, int64_t(1) << desc->log2_T[0],
                    desc->L, 4);
    if (st != HG_OK) return st;
    if ((st = make_common(desc, 1, n, p.c)) != HG_OK) return st;
    if (n == 0 || (!g_gamma && !g_dgamma && !g_lap && !g_stencil)) return ok();
    if (!coords) return fail(HG_ERR_INVALID_ARG, "coords must not be NULL");
    if (!aligned(coords, 4) || (g_gamma && !aligned(g_gamma, 4)) || (g_dgamma && !aligned(g_dgamma, 4)) ||
        (g_lap && !aligned(g_lap, 4)) || (g_stencil && !aligned(g_stencil, 4)))
        return fail(HG_ERR_INVALID_ARG, "coords and upstream gradients must be 4-byte aligned");
    memset(&p.grad, 0, sizeof(p.grad));
    p.grad.ptr[0] = grad->ptr;
    p.grad.ls[0] = grad->level_stride;
    p.grad.rs[0] = grad->row_stride;
    p.coords = coords;
    p.g_gamma = g_gamma;
    p.g_dgamma = g_dgamma;
    p.g_lap = g_lap;
    p.g_hess = nullptr;
    p.g_stencil = g_stencil;
    p.eps = eps;
    const int fc = (F % 2 == 0) ? 2 : 1;
    const bool vec = fc == 2 && aligned(grad->ptr, 8) && grad->row_stride % 2 == 0 && grad->level_stride % 2 == 0;
    // A point adds up to (2d+1) 2^d contributions, so shared-memory atomics cost more than in the
    // d-linear backward: measured on the 3D INGP-FD workload, privatising its 38-140 KB coarse
    // levels made the backward slower (4.77 vs 4.48 ms); only levels of at most 32 KB -- a few
    // thousand rows, where direct REDs serialise -- are privatised.
    plan_backward(p, true, static_cast<int64_t>(F) * 4, 1, kHermitePrivLevelBytes);
    return launch_status(hg::launch_linear_fd_bwd(p, fc, vec, stream), "finite-difference backward");
}

// Gaussian-RBF grid: shared argument checks (the d-linear table's, plus d, eps and rings).
hg_status rbf_check(const hg_grid_desc* desc, int64_t n, float eps, int32_t rings) {
    hg_status st = check_desc(desc, 1);
    if (st != HG_OK) return st;
    if ((st = check_n(n)) != HG_OK) return st;
    if (desc->d > 3) return fail(HG_ERR_UNSUPPORTED, "the Gaussian-RBF grid is built for d = 2 and 3, not %d", desc->d);
    if (!(eps > 0.0f) || !(eps < INFINITY)) return fail(HG_ERR_INVALID_ARG, "eps = %g; must be positive and finite", eps);
    if (rings < 1 || rings > 4) return fail(HG_ERR_INVALID_ARG, "rings = %d; must be in 1..4", rings);
    return HG_OK;
}

hg_status hg_rbf_fwd(const hg_grid_desc* desc, int64_t n, const float* coords, float eps, int32_t rings,
                     const hg_table* table, float* gamma, float* dgamma, float* lap, hg_stream stream) {
    hg_status st = rbf_check(desc, n, eps, rings);
    if (st != HG_OK) return st;
    if (!table) return fail(HG_ERR_INVALID_ARG, "table is NULL");
    const int F = desc->F;
    const size_t es = dtype_size(desc->dtype);
    st = check_view("table", 0, table->ptr, table->level_stride, table->row_stride, F, int64_t(1) << desc->log2_T[0],
                    desc->L, es);
    if (st != HG_OK) return st;
    hg::FwdParams p;
    if ((st = make_common(desc, 1, n, p.c)) != HG_OK) return st;
    if (n == 0) return ok();
    if (!coords || !gamma) return fail(HG_ERR_INVALID_ARG, "coords and gamma must not be NULL");
    if (!aligned(coords, 4) || !aligned(gamma, 4) || (dgamma && !aligned(dgamma, 4)) || (lap && !aligned(lap, 4)))
        return fail(HG_ERR_INVALID_ARG, "coords and outputs must be 4-byte aligned");
    memset(&p.tab, 0, sizeof(p.tab));
    p.tab.ptr[0] = table->ptr;
    p.tab.ls[0] = table->level_stride;
    p.tab.rs[0] = table->row_stride;
    p.coords = coords;
    p.gamma = gamma;
    p.dgamma = dgamma;
    p.lap = lap;
    p.hess = nullptr;
    p.stencil = nullptr;
    p.eps = eps;
    all_levels(p.c);
    return launch_status(hg::launch_rbf_fwd(p, (F % 2 == 0) ? 2 : 1, rings, desc->dtype, stream), "RBF forward");
}

hg_status hg_rbf_bwd(const hg_grid_desc* desc, int64_t n, const float* coords, float eps, int32_t rings,
                     const float* g_gamma, const float* g_dgamma, const float* g_lap, const hg_grad_table* grad,
                     hg_stream stream) {
    hg_status st = rbf_check(desc, n, eps, rings);
    if (st != HG_OK) return st;
    if (!grad) return fail(HG_ERR_INVALID_ARG, "grad is NULL");
    const int F = desc->F;
    st = check_view("grad", 0, grad->ptr, grad->level_stride, grad->row_stride, F, int64_t(1) << desc->log2_T[0],
                    desc->L, 4);
    if (st != HG_OK) return st;
    hg::BwdParams p;
    if ((st = make_common(desc, 1, n, p.c)) != HG_OK) return st;
    if (n == 0 || (!g_gamma && !g_dgamma && !g_lap)) return ok();
    if (!coords) return fail(HG_ERR_INVALID_ARG, "coords must not be NULL");
    if (!aligned(coords, 4) || (g_gamma && !aligned(g_gamma, 4)) || (g_dgamma && !aligned(g_dgamma, 4)) ||
        (g_lap && !aligned(g_lap, 4)))
        return fail(HG_ERR_INVALID_ARG, "coords and upstream gradients must be 4-byte aligned");
    memset(&p.grad, 0, sizeof(p.grad));
    p.grad.ptr[0] = grad->ptr;
    p.grad.ls[0] = grad->level_stride;
    p.grad.rs[0] = grad->row_stride;
    p.coords = coords;
    p.g_gamma = g_gamma;
    p.g_dgamma = g_dgamma;
    p.g_lap = g_lap;
    p.g_hess = nullptr;
    p.g_stencil = nullptr;
    p.eps = eps;
    const int fc = (F % 2 == 0) ? 2 : 1;
    const bool vec = fc == 2 && aligned(grad->ptr, 8) && grad->row_stride % 2 == 0 && grad->level_stride % 2 == 0;
    all_levels(p.c);  // every level takes the tiled kernel (a CTA's tile covers its points' taps)
    const bool any = p.c.level_mask != 0;
    if (!any) return ok();
    return launch_status(hg::launch_rbf_bwd(p, fc, vec, rings, stream), "RBF backward");
}

hg_status hg_hash_indices(const hg_grid_desc* desc, int64_t n, const float* coords, uint32_t* idx, hg_stream stream) {
    hg_status st = check_desc(desc, desc ? desc->d + 1 : 0);
    if (st != HG_OK) return st;
    if ((st = check_n(n)) != HG_OK) return st;
    hg::IdxParams p;
    if ((st = make_common(desc, desc->d + 1, n, p.c)) != HG_OK) return st;
    if (n == 0) return ok();
    if (!coords || !idx) return fail(HG_ERR_INVALID_ARG, "coords and idx must not be NULL");
    if (!aligned(coords, 4) || !aligned(idx, 4)) return fail(HG_ERR_INVALID_ARG, "coords and idx must be 4-byte aligned");
    p.coords = coords;
    p.idx = idx;
    all_levels(p.c);
    return launch_status(hg::launch_indices(p, stream), "vertex indices");
}

hg_status hg_probe_replay_gather(const hg_grid_desc* desc, int64_t n, const float* coords, const void* table,
                                 int64_t level_stride_bytes, int32_t row_bytes, int32_t lanes_per_row, float* sink,
                                 hg_stream stream) {
    return replay(desc, n, coords, const_cast<void*>(table), level_stride_bytes, row_bytes, lanes_per_row, sink, false,
                  stream);
}

hg_status hg_probe_replay_red(const hg_grid_desc* desc, int64_t n, const float* coords, float* grad,
                              int64_t level_stride_bytes, int32_t row_bytes, int32_t lanes_per_row, hg_stream stream) {
    return replay(desc, n, coords, grad, level_stride_bytes, row_bytes, lanes_per_row, nullptr, true, stream);
}


hg_status hg_siren_fwd(const hg_siren_desc* desc, int64_t n, const float* gamma, const float* dgamma,
                       const float* lap, const float* W1, const float* b1, const float* W2, const float* b2,
                       float* u, float* du, float* lapu, hg_stream stream) {
    hg::SirenParams p;
    int ctas = 0;
    hg_status st = siren_plan(desc, n, p);
    if (st != HG_OK) return st;
    if (!gamma || !W1 || !b1 || !W2) return fail(HG_ERR_INVALID_ARG, "gamma, W1, b1 and W2 must not be NULL");
    if ((du || lapu) && !dgamma) return fail(HG_ERR_INVALID_ARG, "du and lapu need dgamma");
    if (lapu && !lap) return fail(HG_ERR_INVALID_ARG, "lapu needs lap");
    const void* ptrs[] = {gamma, dgamma, lap, W1, b1, W2, b2, u, du, lapu};
    for (const void* q : ptrs)
        if (q && !aligned(q, 4)) return fail(HG_ERR_INVALID_ARG, "pointers must be 4-byte aligned");
    if (n == 0 || (!u && !du && !lapu)) return ok();
    p.in[0] = gamma;
    for (int i = 0; i < p.d; ++i) p.in[1 + i] = dgamma ? dgamma + static_cast<int64_t>(i) * p.K * n : nullptr;
    p.in[p.d + 1] = lap;
    p.W1 = W1;
    p.b1 = b1;
    p.W2 = W2;
    p.b2 = b2;
    p.u = u;
    p.du = du;
    p.lapu = lapu;
    int smem_max = 0;
    if (query_smem_max(smem_max) != HG_OK) return fail(HG_ERR_CUDA, "device query failed");
    if (hg::siren_tc_usable(p, smem_max))
        return launch_status(hg::launch_siren_fwd_tc(p, stream), "SIREN forward (tensor cores)");
    if ((st = siren_grid(p, false, ctas)) != HG_OK) return st;
    return launch_status(hg::launch_siren_fwd(p, ctas, stream), "SIREN forward");
}

hg_status hg_encode_siren_fwd(const hg_grid_desc* desc, int64_t n, const float* coords, const hg_table* tables,
                              const hg_siren_desc* sdesc, const float* W1, const float* b1, const float* W2,
                              const float* b2, float* u, float* du, float* lapu, hg_stream stream) {
    hg_status st = check_desc(desc, desc ? desc->d + 1 : 0);
    if (st != HG_OK) return st;
    if ((st = check_n(n)) != HG_OK) return st;
    if (!tables) return fail(HG_ERR_INVALID_ARG, "tables is NULL");
    if (desc->d != 2 && desc->d != 3)
        return fail(HG_ERR_UNSUPPORTED, "the fused encoder + SIREN forward takes d = 2 or 3 (got %d)", desc->d);
    if (desc->F != 2) return fail(HG_ERR_UNSUPPORTED, "the fused encoder + SIREN forward takes F = 2 (got %d)", desc->F);
    hg::SirenParams p;
    if ((st = siren_plan(sdesc, n, p)) != HG_OK) return st;
    if (sdesc->d != desc->d)
        return fail(HG_ERR_INVALID_ARG, "the SIREN's d = %d differs from the grid's d = %d", sdesc->d, desc->d);
    if (sdesc->K != desc->L * desc->F)
        return fail(HG_ERR_INVALID_ARG, "the SIREN's K = %d must be L * F = %d", sdesc->K, desc->L * desc->F);
    const int d = desc->d, F = desc->F, V = 1 << d;
    const size_t es = dtype_size(desc->dtype);
    const void* ptrs[5];
    int64_t ls[5], rs[5];
    for (int k = 0; k <= d; ++k) {
        ptrs[k] = tables[k].ptr;
        ls[k] = tables[k].level_stride;
        rs[k] = tables[k].row_stride;
        st = check_view("tables", k, ptrs[k], ls[k], rs[k], static_cast<int64_t>(binom(d, k)) * F,
                        int64_t(1) << desc->log2_T[k], desc->L, es);
        if (st != HG_OK) return st;
    }
    const size_t row = static_cast<size_t>(V) * F * es;
    const size_t al = row < 32 ? row : 32;
    if (!is_packed(desc, ptrs, ls, rs, es) || !aligned(ptrs[0], al) || (static_cast<size_t>(ls[0]) * es) % al != 0)
        return fail(HG_ERR_UNSUPPORTED, "the fused encoder + SIREN forward needs the packed table layout, "
                                        "%zu-byte aligned", al);
    if (!W1 || !b1 || !W2) return fail(HG_ERR_INVALID_ARG, "W1, b1 and W2 must not be NULL");
    const void* vp[] = {coords, W1, b1, W2, b2, u, du, lapu};
    for (const void* q : vp)
        if (q && !aligned(q, 4)) return fail(HG_ERR_INVALID_ARG, "pointers must be 4-byte aligned");
    if (n == 0 || (!u && !du && !lapu)) return ok();
    if (!coords) return fail(HG_ERR_INVALID_ARG, "coords must not be NULL");
    hg::FwdParams e;
    memset(&e, 0, sizeof(e));
    if ((st = make_common(desc, d + 1, n, e.c)) != HG_OK) return st;
    for (int k = 0; k <= d; ++k) {
        e.tab.ptr[k] = ptrs[k];
        e.tab.ls[k] = ls[k];
        e.tab.rs[k] = rs[k];
    }
    e.coords = coords;
    all_levels(e.c);
    p.W1 = W1;
    p.b1 = b1;
    p.W2 = W2;
    p.b2 = b2;
    p.u = u;
    p.du = du;
    p.lapu = lapu;
    p.nbuf = 1;  // the tile is computed in place, not copied
    int dev = 0, sms = 0, smem_max = 0, per_sm = 0;
    cudaError_t ce = cudaGetDevice(&dev);
    if (ce == cudaSuccess) ce = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (ce == cudaSuccess) ce = cudaDeviceGetAttribute(&smem_max, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (ce != cudaSuccess) return fail(HG_ERR_CUDA, "device query failed: %s", cudaGetErrorString(ce));
    const size_t bytes = hg::siren_smem_bytes(p, false);
    if (bytes > static_cast<size_t>(smem_max))
        return fail(HG_ERR_UNSUPPORTED, "a SIREN tile needs %zu bytes of shared memory (at most %d)", bytes, smem_max);
    ce = static_cast<cudaError_t>(hg::encode_siren_ctas_per_sm(p, desc->dtype, &per_sm));
    if (ce != cudaSuccess || per_sm < 1) return fail(HG_ERR_CUDA, "fused encoder + SIREN occupancy query failed");
    const int64_t tiles = (n + p.pts - 1) / p.pts;
    const int ctas = static_cast<int>(std::min<int64_t>(tiles, static_cast<int64_t>(sms) * per_sm));
    return launch_status(hg::launch_encode_siren_fwd(p, e, desc->dtype, ctas, stream), "fused encoder + SIREN forward");
}

hg_status hg_siren_bwd(const hg_siren_desc* desc, int64_t n, const float* gamma, const float* dgamma,
                       const float* lap, const float* W1, const float* b1, const float* W2, const float* g_u,
                       const float* g_du, const float* g_lapu, float* g_gamma, float* g_dgamma, float* g_lap,
                       float* gW1, float* gb1, float* gW2, float* gb2, hg_stream stream) {
    hg::SirenParams p;
    int ctas = 0;
    hg_status st = siren_plan(desc, n, p);
    if (st != HG_OK) return st;
    if (!gamma || !dgamma || !lap || !W1 || !b1 || !W2)
        return fail(HG_ERR_INVALID_ARG, "gamma, dgamma, lap, W1, b1 and W2 must not be NULL");
    const void* ptrs[] = {gamma, dgamma, lap, W1, b1, W2, g_u, g_du, g_lapu, g_gamma, g_dgamma, g_lap,
                          gW1, gb1, gW2, gb2};
    for (const void* q : ptrs)
        if (q && !aligned(q, 4)) return fail(HG_ERR_INVALID_ARG, "pointers must be 4-byte aligned");
    if (n == 0 || (!g_gamma && !g_dgamma && !g_lap && !gW1 && !gb1 && !gW2 && !gb2)) return ok();
    const int64_t row = static_cast<int64_t>(p.K) * n;
    p.in[0] = gamma;
    p.g_in[0] = g_gamma;
    for (int i = 0; i < p.d; ++i) {
        p.in[1 + i] = dgamma + i * row;
        p.g_in[1 + i] = g_dgamma ? g_dgamma + i * row : nullptr;
    }
    p.in[p.d + 1] = lap;
    p.g_in[p.d + 1] = g_lap;
    p.W1 = W1;
    p.b1 = b1;
    p.W2 = W2;
    p.g_u = g_u;
    p.g_du = g_du;
    p.g_lapu = g_lapu;
    p.gW1 = gW1;
    p.gb1 = gb1;
    p.gW2 = gW2;
    p.gb2 = gb2;
    hg::siren_bwd_tiles(p);
    if ((st = siren_grid(p, true, ctas)) != HG_OK) return st;
    return launch_status(hg::launch_siren_bwd(p, ctas, stream), "SIREN backward");
}

}  // extern "C"
