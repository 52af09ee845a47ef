/*
 * hg.h -- C ABI of the B300 multiresolution hash-grid encoding library
 * (libhg.so, built for sm_103a).
 *
 * The library evaluates the gradient-augmented cubic-Hermite hash encoding
 * (Hermite-NGP) -- per query point and level the encoding gamma, its spatial
 * gradient and its Laplacian in one pass -- together with its backward
 * scatter into the coefficient tables, and the plain d-linear Instant-NGP
 * encoding as the degenerate case.
 *
 * Sources (page title, section):
 *   [HNGP]  "Hermite-NGP: Gradient-Augmented Hash Encoding for Learning PDEs":
 *           整体框架 (the pipeline), 关键设计 1 (encoding equation, bases,
 *           order-bucketed tables), 关键设计 2 (analytic gradient and
 *           Laplacian), 关键设计 3 (coarse-to-fine active levels),
 *           消融实验 (per-order table sizes 14-14-10 / 12-12-12 / 14-10-14).
 *   [INGP]  "SIGGRAPH 2022｜InstantNGP 与多分辨率哈希编码": 流程与原理
 *           (steps 1-4: corner lookup, hashing, d-linear interpolation, level
 *           concatenation; one-to-one vs hashed levels).
 *   [NEWS]  "英偉達將訓練 NeRF 模型從 5 小時縮至 5 秒": the geometric progression
 *           of level resolutions between N_min and N_max; hashed levels whose
 *           colliding gradients add up; control-flow-free parallel lookups.
 *
 * Conventions shared by every entry point:
 *   - Memory: every pointer argument except `desc`, `desc->res`, `res_out`
 *     and the arrays of table descriptors is a DEVICE pointer owned by the
 *     caller.  The library allocates no device memory and keeps no state
 *     between calls.
 *   - Asynchrony: kernels are enqueued on `stream` (NULL = legacy default
 *     stream); no call synchronises.  Argument checking is synchronous: on
 *     any error status nothing has been enqueued.  Launch errors are reported
 *     as HG_ERR_CUDA (asynchronous execution faults surface at the caller's
 *     next synchronisation, as usual in CUDA).
 *   - Errors: every call returns an hg_status; hg_last_error() returns a
 *     human-readable reason for the last failure on the calling thread.
 *     No C++ exception crosses the ABI.
 *   - Points: coords is float32 [n][d], row-major (AoS).  A coordinate is
 *     clamped to [0,1] (NaN reads as 0).
 *   - Levels: resolution N_l, vertex spacing dx_l = 1/N_l; the level's grid
 *     has N_l+1 vertices per axis.  pos = fl32(x * N_l) (one fp32 multiply,
 *     round to nearest), cell c = min(floor(pos), N_l - 1), local coordinate
 *     t = pos - c in [0,1].
 *   - Dimension d = 2, 3 or 4.  The 4D (space-time) grid is the extension
 *     [HNGP 局限与展望] names as the method's main storage cost: 16
 *     coefficients per vertex and feature, same equation.
 *   - Vertex index in order table k (size T_k = 2^log2_T[k]): when the
 *     level's (N_l+1)^d vertices fit in T_k the index is one-to-one,
 *     sum_i g_i (N_l+1)^i; otherwise it is the spatial hash
 *     (g_0 * 1 XOR g_1 * 2654435761 [XOR g_2 * 805459861 [XOR g_3 * 3674653429]])
 *     mod 2^32 mod T_k.  [INGP 流程与原理; NEWS; the pages print no hash
 *     formula: these are Instant-NGP's published primes, in order]
 *   - Corners of a cell are numbered v = sum_i v_i 2^i (bit i = axis i).
 *   - Multi-indices alpha in {0,1}^d (bit i = d/dx_i) are bucketed by order
 *     k = |alpha| into d+1 tables [HNGP 关键设计 1]; inside bucket k they are
 *     ordered lexicographically by axis list (3D: k=1 x,y,z; k=2 xy,xz,yz;
 *     k=3 xyz; 4D: k=1 x,y,z,w; k=2 xy,xz,xw,yz,yw,zw; k=3 xyz,xyw,xzw,yzw;
 *     k=4 xyzw), and each entry of table k holds C(d,k)*F values,
 *     alpha-major, feature-minor.
 *   - Outputs and upstream gradients are float32 in one of two layouts
 *     (hg_layout):
 *       HG_POINT_MAJOR:   gamma, lap [n][L][F]; dgamma [n][d][L][F]
 *       HG_FEATURE_MAJOR: gamma, lap [L][F][n]; dgamma [d][L][F][n]
 *     Feature-major is the column-major [n x L*F] matrix a following GEMM
 *     reads directly, and is the layout the kernels write fastest.
 *   - Inactive levels (bit l of level_mask clear) are written as zeros by
 *     the forwards and receive no gradient [HNGP 关键设计 3].
 */
#ifndef HG_H
#define HG_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t / CUstream. */
typedef struct CUstream_st* hg_stream;

typedef enum {
    HG_OK = 0,
    HG_ERR_INVALID_ARG = 1,   /* a value out of range, a NULL that may not be NULL */
    HG_ERR_UNSUPPORTED = 2,   /* a valid request this build does not implement */
    HG_ERR_CUDA = 3           /* a CUDA runtime call or kernel launch failed */
} hg_status;

typedef enum { HG_F32 = 0, HG_F16 = 1 } hg_dtype;
typedef enum { HG_POINT_MAJOR = 0, HG_FEATURE_MAJOR = 1 } hg_layout;

#define HG_MAX_LEVELS 32
#define HG_MAX_RESOLUTION (1 << 22)
#define HG_MAX_LOG2_T 30

/* Grid description (host memory, read during the call only). */
typedef struct {
    int32_t d;              /* spatial dimension: 2, 3 or 4 */
    int32_t L;              /* number of levels: 1..32 */
    int32_t F;              /* features per level: 1, 2, 4 or 8 */
    int32_t n_min, n_max;   /* level schedule (see hg_level_resolutions);
                               ignored when res != NULL */
    const int32_t* res;     /* optional host array [L] of explicit resolutions,
                               each in 1..HG_MAX_RESOLUTION */
    int32_t log2_T[5];      /* entries per level of order table k = 0..d
                               (0..HG_MAX_LOG2_T); the d-linear calls use
                               log2_T[0] only */
    uint32_t level_mask;    /* bit l set = level l active; bits >= L must be 0 */
    int32_t dtype;          /* hg_dtype of the coefficient tables */
    int32_t layout;         /* hg_layout of outputs and upstream gradients */
} hg_grid_desc;

/* A read-only coefficient table view: element (level l, entry i, value j)
 * is at ptr + l*level_stride + i*row_stride + j (strides in ELEMENTS of the
 * table dtype).  Rows must not overlap: row_stride >= values per entry and,
 * when L > 1, level_stride >= T*row_stride.  Views of different orders may
 * interleave inside one buffer (the "packed" layout below). */
typedef struct {
    const void* ptr;
    int64_t level_stride;
    int64_t row_stride;
} hg_table;

/* A float32 gradient table view, same indexing; accumulated with +=. */
typedef struct {
    float* ptr;
    int64_t level_stride;
    int64_t row_stride;
} hg_grad_table;

/* Packed (interleaved) layout -- the fast path.  When all T_k are equal, one
 * buffer [L][T][2^d][F] holds every order with a vertex's 2^d slots ordered
 * by order, then as in the buckets: 2D (f, fx, fy, fxy); 3D (f, fx, fy, fz,
 * fxy, fxz, fyz, fxyz); 4D (f, fx, fy, fz, fw, fxy, fxz, fxw, fyz, fyw, fzw,
 * fxyz, fxyw, fxzw, fyzw, fxyzw); table k is then the view
 * ptr + off_k*F, row_stride 2^d*F, level_stride T*2^d*F, with
 * off_k = sum_{k'<k} C(d,k').  The library detects this layout (and 16-byte
 * alignment) and reads or scatters a vertex's whole row with vector accesses;
 * any other layout takes the element-wise path of the same kernels. */

/* ------------------------------------------------------------------------ */

/* Level schedule [NEWS, geometric progression; the printed formula is lost
 * in the page's extraction]: N_l = floor(n_min * b^l), b = (n_max/n_min)^(1/(L-1)),
 * evaluated exactly (N_l is the largest n with
 * n^(L-1) * n_min^l <= n_max^l * n_min^(L-1)), so N_0 = n_min and
 * N_{L-1} = n_max.  L = 1 gives N_0 = n_min.  If desc->res is set, copies it.
 * res_out: host array [desc->L].  Host only; enqueues nothing.
 * Errors: HG_ERR_INVALID_ARG for a NULL pointer, L out of 1..32,
 * n_min < 1, n_max < n_min or n_max > HG_MAX_RESOLUTION. */
hg_status hg_level_resolutions(const hg_grid_desc* desc, int32_t* res_out);

/* Hermite forward [HNGP 整体框架, 关键设计 1, 关键设计 2]: for every point and
 * active level,
 *   gamma   = sum_{corner g} sum_{alpha} theta^(alpha)[idx_k(g)] H^(alpha)((x - x_g)/dx) dx^|alpha|
 *   dgamma_j = d gamma / d x_j,  lap = sum_j d^2 gamma / d x_j^2,
 * with H^(alpha) = prod_i h^(alpha_i), the cubic Hermite value basis
 * (h^(0)) and slope basis (h^(1)) of each corner.
 *   n:       number of points (0 is a no-op), n <= 2^31 - 1
 *   coords:  device float32 [n][d]
 *   tables:  host array [d+1] of order-table views (dtype desc->dtype);
 *            table k has T_k entries of C(d,k)*F values per level
 *   gamma:   device float32 output (required when n > 0)
 *   dgamma:  device float32 output or NULL (not computed)
 *   lap:     device float32 output or NULL (not computed)
 * Arithmetic is fp32 (fp16 coefficients are widened exactly).
 * Errors: HG_ERR_INVALID_ARG (bad descriptor, NULL required pointer,
 * overlapping rows), HG_ERR_CUDA (launch failure). */
hg_status hg_encode_fwd(const hg_grid_desc* desc, int64_t n, const float* coords,
                        const hg_table* tables, float* gamma, float* dgamma, float* lap,
                        hg_stream stream);

/* Hermite backward [HNGP 整体框架 flowchart: backpropagation updates the hash
 * coefficients; NEWS: colliding entries' gradients add up]: the transpose of
 * hg_encode_fwd.  For every point, active level, corner and alpha,
 *   grad_k[l][idx_k(g)][slot(alpha)][f] +=
 *       dx^|alpha| * ( g_gamma * H + sum_j g_dgamma_j * dH/dx_j
 *                                  + g_lap * sum_j d^2H/dx_j^2 ).
 *   g_gamma, g_dgamma, g_lap: device float32 upstream gradients in the
 *            layout of the forward's outputs; any of them may be NULL
 *            (treated as zero)
 *   grads:   host array [d+1] of float32 gradient-table views, accumulated
 *            with atomic adds (the caller zeroes them); the order in which
 *            colliding contributions add is unspecified, so results agree
 *            with an exact sum to rounding, not bit for bit.
 * Errors: as hg_encode_fwd. */
hg_status hg_encode_bwd(const hg_grid_desc* desc, int64_t n, const float* coords,
                        const float* g_gamma, const float* g_dgamma, const float* g_lap,
                        const hg_grad_table* grads, hg_stream stream);

/* Hermite forward with the full Hessian: the second derivatives of the
 * encoding's bases [HNGP 关键设计 2] give every d2 gamma / dx_i dx_j, not only
 * their sum (the Laplacian), for PDEs with mixed derivatives.  For each point
 * and active level the P = d(d+1)/2 entries of the upper triangle, row-major
 * (2D xx, xy, yy; 3D xx, xy, xz, yy, yz, zz), are
 *   hess_ij = sum_g sum_alpha theta^(alpha)[idx_k(g)] dx^|alpha| d2H/dx_i dx_j.
 *   gamma, dgamma: as hg_encode_fwd (dgamma may be NULL)
 *   hess:   device float32 output (required when n > 0):
 *           HG_POINT_MAJOR [n][P][L][F], HG_FEATURE_MAJOR [P][L][F][n]
 * The trace of hess equals hg_encode_fwd's lap to rounding.
 * Errors: as hg_encode_fwd. */
hg_status hg_encode_fwd_hessian(const hg_grid_desc* desc, int64_t n, const float* coords,
                                const hg_table* tables, float* gamma, float* dgamma, float* hess,
                                hg_stream stream);

/* Backward of hg_encode_fwd_hessian: as hg_encode_bwd with the upstream
 * gradient of the Hessian (g_hess, the layout of hess, may be NULL) in place
 * of that of the Laplacian:
 *   grad_k[l][idx_k(g)][slot(alpha)][f] += dx^|alpha| * ( g_gamma * H
 *       + sum_j g_dgamma_j * dH/dx_j + sum_{i<=j} g_hess_ij * d2H/dx_i dx_j ).
 * Errors: as hg_encode_fwd. */
hg_status hg_encode_bwd_hessian(const hg_grid_desc* desc, int64_t n, const float* coords,
                                const float* g_gamma, const float* g_dgamma, const float* g_hess,
                                const hg_grad_table* grads, hg_stream stream);

/* d-linear forward (Instant-NGP) [INGP 流程与原理 steps 1-3]:
 *   gamma[l][f] = sum_{corner v} w_v * table[l][idx_0(c+v)][f],
 *   w_v = prod_i (v_i ? t_i : 1 - t_i),
 * with one table of T = 2^log2_T[0] entries of F values per level.
 *   table: host pointer to ONE view (dtype desc->dtype)
 *   gamma: device float32 output in desc->layout (the gamma shape above)
 * Errors: as hg_encode_fwd. */
hg_status hg_linear_fwd(const hg_grid_desc* desc, int64_t n, const float* coords,
                        const hg_table* table, float* gamma, hg_stream stream);

/* d-linear backward: grad[l][idx_0(c+v)][f] += w_v * g_gamma[l][f]
 * (atomic adds; the caller zeroes grad).  grad: host pointer to ONE float32
 * view.  Errors: as hg_encode_fwd. */
hg_status hg_linear_bwd(const hg_grid_desc* desc, int64_t n, const float* coords,
                        const float* g_gamma, const hg_grad_table* grad, hg_stream stream);

/* INGP-FD: the d-linear encoding with central finite differences -- the
 * finite-difference baseline [HNGP 研究背景与动机, 关键设计 2] that takes the
 * Laplacian from 2d+1 d-linear encodes.  For every point and active level,
 * with the stencil points x + eps e_i and x - eps e_i (each shifted
 * coordinate is one fp32 add, x_i + eps or x_i - eps, then clamped and
 * located as in hg_linear_fwd):
 *   gamma    = gamma(x)                                     [n][L][F] / [L][F][n]
 *   dgamma_i = (gamma(x + eps e_i) - gamma(x - eps e_i)) / (2 eps)
 *   lap      = sum_i (gamma(x + eps e_i) - 2 gamma(x) + gamma(x - eps e_i)) / eps^2
 *   stencil_j = gamma at stencil point j (j = 2i: x + eps e_i; j = 2i + 1:
 *              x - eps e_i): HG_POINT_MAJOR [n][2d][L][F], HG_FEATURE_MAJOR
 *              [2d][L][F][n] -- the encodings INGP-FD feeds its network.
 *   eps:     the step, positive and finite (1/eps^2 must not overflow fp32)
 *   table:   as hg_linear_fwd (one table, log2_T[0])
 *   gamma:   device float32 output (required when n > 0)
 *   dgamma, lap, stencil: device float32 outputs or NULL (not computed)
 * Arithmetic fp32 (the factors 1/(2 eps) and 1/eps^2 rounded once).
 * Errors: as hg_linear_fwd; HG_ERR_INVALID_ARG for a bad eps. */
hg_status hg_linear_fd_fwd(const hg_grid_desc* desc, int64_t n, const float* coords, float eps,
                           const hg_table* table, float* gamma, float* dgamma, float* lap, float* stencil,
                           hg_stream stream);

/* Backward of hg_linear_fd_fwd: every stencil point scatters, with its
 * d-linear corner weights, the upstream weight of its value in the outputs,
 *   x:            g_gamma - (2d / eps^2) g_lap
 *   x + eps e_i:  g_dgamma_i / (2 eps) + g_lap / eps^2 + g_stencil_2i
 *   x - eps e_i: -g_dgamma_i / (2 eps) + g_lap / eps^2 + g_stencil_2i+1
 * into the fp32 gradient table `grad` (accumulated, caller-zeroed).  Upstream
 * gradients in the layouts of the forward's outputs; any may be NULL.
 * Errors: as hg_linear_bwd; HG_ERR_INVALID_ARG for a bad eps. */
hg_status hg_linear_fd_bwd(const hg_grid_desc* desc, int64_t n, const float* coords, float eps,
                           const float* g_gamma, const float* g_dgamma, const float* g_lap,
                           const float* g_stencil, const hg_grad_table* grad, hg_stream stream);

/* Gaussian-RBF multi-resolution grid (DInf-Grid) ["DInf-Grid：一种基于可微特征网格的
 * 神经微分方程求解器", 可微的径向基函数插值, 多分辨率特征网格]: per point and active
 * level, the features interpolated with normalised Gaussian weights over a
 * ring neighbourhood of the point's cell,
 *   gamma = sum_g w_g F_g,  w_g = phi(|y - g|) / sum_h phi(|y - h|),  phi(r) = exp(-(eps r)^2),
 * with y = pos = fl32(x * N_l) the point in grid units (vertex g at y = g),
 * the neighbourhood the box c_i - rings + 1 <= g_i <= c_i + rings clipped
 * to the grid (0 <= g_i <= N_l), and dgamma, lap its exact gradient and
 * Laplacian in x.  Vertices are indexed as in hg_linear_fwd (one-to-one
 * when the level's (N_l+1)^d vertices fit T = 2^log2_T[0] -- the page's
 * dense grids -- hashed otherwise); the table is [L][T][F] like the
 * d-linear one.  Outputs as hg_encode_fwd (dgamma, lap may be NULL).
 *   eps:   kernel width in grid units, positive and finite (the page: 1)
 *   rings: 1..4 (the page: 3 for eps = 1)
 * Arithmetic fp32.  Errors: as hg_linear_fwd; HG_ERR_INVALID_ARG for a bad
 * eps or rings; HG_ERR_UNSUPPORTED for d = 4. */
hg_status hg_rbf_fwd(const hg_grid_desc* desc, int64_t n, const float* coords, float eps, int32_t rings,
                     const hg_table* table, float* gamma, float* dgamma, float* lap, hg_stream stream);

/* Backward of hg_rbf_fwd: grad[l][idx(g)][f] += g_gamma w_g + sum_j g_dgamma_j
 * dw_g/dx_j + g_lap lap w_g for every tap g, into the fp32 table `grad`
 * (accumulated, caller-zeroed).  Errors: as hg_rbf_fwd. */
hg_status hg_rbf_bwd(const hg_grid_desc* desc, int64_t n, const float* coords, float eps, int32_t rings,
                     const float* g_gamma, const float* g_dgamma, const float* g_lap, const hg_grad_table* grad,
                     hg_stream stream);

/* SIREN chain-rule consumer of the encoding ["Hermite-NGP: Gradient-Augmented
 * Hash Encoding for Learning PDEs", 整体框架 (grad u = du/dgamma grad gamma,
 * lap u = d2u/dgamma2 (grad gamma)^2 + du/dgamma lap gamma) and 关键设计 2
 * (SIREN, sigma = sin(omega .), one-layer Laplacian)]:
 *   z = W1 gamma + b1,  a = sin(omega z),  y_i = W1 dgamma/dx_i,  s = W1 lap gamma,
 *   u = W2 a + b2,  du/dx_i = W2 (omega cos(omega z) * y_i),
 *   lap u = W2 (omega cos(omega z) * s - omega^2 a * sum_i y_i^2).
 * The inputs are the encoding's outputs in its feature-major layout with the
 * levels' features concatenated (K = L F): gamma [K][n], dgamma [d][K][n],
 * lap [K][n]. */
typedef struct {
    int32_t d;      /* spatial dimensions of the derivatives, 1..4 */
    int32_t K;      /* inputs per point (L F), a multiple of 8 up to 64 */
    int32_t H;      /* hidden width: 16, 32, 64 or 128 */
    int32_t O;      /* outputs, 1..4 */
    float omega;    /* frequency of the sine layer (omega_0 = 30 on the page), finite */
} hg_siren_desc;

/* Forward.  Device pointers, fp32, all 4-byte aligned: gamma [K][n];
 * dgamma [d][K][n] (needed for du or lapu, else may be NULL); lap [K][n]
 * (needed for lapu); W1 [H][K], b1 [H], W2 [O][H] row-major, b2 [O] (NULL =
 * zero).  Outputs (written; each may be NULL): u [O][n], du [d][O][n],
 * lapu [O][n].  Arithmetic fp32.  Errors: HG_ERR_INVALID_ARG for NULL
 * required pointers, a bad desc or n outside 0..2^31-1; HG_ERR_UNSUPPORTED
 * when a CTA's tile does not fit in shared memory; HG_ERR_CUDA on a launch
 * failure. */
hg_status hg_siren_fwd(const hg_siren_desc* desc, int64_t n, const float* gamma, const float* dgamma,
                       const float* lap, const float* W1, const float* b1, const float* W2, const float* b2,
                       float* u, float* du, float* lapu, hg_stream stream);

/* Fused encoder + SIREN forward [HNGP 整体框架: the encoding feeds the
 * network; 关键设计 2: the SIREN chain rule]: u, grad u and lap u of the
 * SIREN at the Hermite encoding of each point, with the encoding (gamma,
 * grad gamma, lap gamma of every level, as hg_encode_fwd computes them)
 * formed on chip and fed to the first layer without being written to
 * memory.  The result equals hg_encode_fwd followed by hg_siren_fwd on its
 * feature-major outputs.  Grid: desc as for hg_encode_fwd with d = 2 or 3,
 * F = 2, the packed table layout (see below; 32-byte aligned rows, 16 bytes
 * for 2D fp16), fp32 or fp16 coefficients; desc->layout is not used (no
 * encoder output is written).  Inactive levels (level_mask) feed zeros.
 * SIREN: sdesc->d = desc->d, sdesc->K = L * F (the levels' features
 * concatenated in level-major, feature-minor order); W1, b1, W2, b2 and the
 * outputs u [O][n], du [d][O][n], lapu [O][n] (each may be NULL) as for
 * hg_siren_fwd.  Device pointers owned by the caller; nothing is allocated.
 * Errors: HG_ERR_INVALID_ARG for a bad desc/sdesc, mismatched d or K, NULL
 * required pointers or n outside 0..2^31-1; HG_ERR_UNSUPPORTED for d, F or
 * a table layout outside the above, or a tile that does not fit in shared
 * memory; HG_ERR_CUDA on a launch failure. */
hg_status hg_encode_siren_fwd(const hg_grid_desc* desc, int64_t n, const float* coords, const hg_table* tables,
                              const hg_siren_desc* sdesc, const float* W1, const float* b1, const float* W2,
                              const float* b2, float* u, float* du, float* lapu, hg_stream stream);

/* Backward: the vector-Jacobian product of hg_siren_fwd with upstream
 * gradients g_u [O][n], g_du [d][O][n], g_lapu [O][n] (NULL = zero).
 * Inputs gamma, dgamma, lap, W1, b1, W2 as for the forward (all required).
 * Input gradients (written; NULL = not wanted): g_gamma [K][n], g_dgamma
 * [d][K][n], g_lap [K][n] -- the upstream gradients of the encoding's
 * backward.  Weight gradients (ACCUMULATED with +=, caller-zeroed; NULL =
 * not wanted): gW1 [H][K], gb1 [H], gW2 [O][H], gb2 [O].  Errors: as
 * hg_siren_fwd. */
hg_status hg_siren_bwd(const hg_siren_desc* desc, int64_t n, const float* gamma, const float* dgamma,
                       const float* lap, const float* W1, const float* b1, const float* W2, const float* g_u,
                       const float* g_du, const float* g_lapu, float* g_gamma, float* g_dgamma, float* g_lap,
                       float* gW1, float* gb1, float* gW2, float* gb2, hg_stream stream);

/* Vertex indices, for checking the lookup bit for bit: idx is device uint32
 * [n][L][d+1][2^d], the index of corner v in order table k at level l, for
 * every level (level_mask does not apply).  Errors: as hg_encode_fwd. */
hg_status hg_hash_indices(const hg_grid_desc* desc, int64_t n, const float* coords,
                          uint32_t* idx, hg_stream stream);

/* Static string naming a status code. */
const char* hg_status_string(hg_status status);

/* Reason for the most recent failing call on this thread ("" if none). */
const char* hg_last_error(void);

/* ABI version of this header (bumped on any incompatible change; 2: log2_T
 * has five entries, d may be 4; 3: the SIREN consumer; 4: the fused encoder
 * + SIREN forward). */
#define HG_ABI_VERSION 4
int32_t hg_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* HG_H */
