// Kernel parameter blocks shared by the C-ABI layer and the kernels.
// Passed by value as __grid_constant__ kernel parameters.
#pragma once

#include <stdint.h>

#include "../../include/hg.h"

namespace hg {

// Per-level constants, computed once per call on the host.
struct Level {
    uint32_t N;       // resolution N_l
    uint32_t side;    // N_l + 1 (vertices per axis)
    uint32_t side2;   // (N_l + 1)^2
    uint32_t dense;   // bit k: order-k table is indexed one-to-one at this level
    float fN;         // (float)N_l      -- d/dx = N d/dt
    float fN2;        // (float)N_l^2
    float dx;         // fp32(1/N_l)     -- the dx^|alpha| scaling
    uint32_t side3;   // (N_l + 1)^3 (only used when a 4D level is one-to-one)
};

struct Common {
    int32_t d, L, F;
    uint32_t level_mask;
    int64_t n;
    uint32_t tmask[5];          // T_k - 1
    // output / upstream-gradient addressing, in elements:
    //   gamma, lap:  n*sn  + (l*F + f)*sf
    //   dgamma:      n*dsn + j*dsj + (l*F + f)*dsf
    //   hess:        n*hsn + q*hsq + (l*F + f)*hsf   (q: upper-triangle entry)
    //   stencil:     n*ssn + j*ssj + (l*F + f)*ssf   (j: finite-difference stencil point, 2d of them)
    int64_t sn, sf, dsn, dsj, dsf, hsn, hsq, hsf, ssn, ssj, ssf;
    Level lv[HG_MAX_LEVELS];
    // levels this launch covers: blockIdx.y -> level lvl[blockIdx.y], nlvl of them
    int32_t nlvl;
    uint8_t lvl[HG_MAX_LEVELS];
};

// Backward levels accumulated in shared memory first (privatised): small
// one-to-one levels whose gradient rows fit one CTA's shared memory.
struct Priv {
    int32_t n;                       // number of privatised levels (grid.y)
    uint8_t lvl[HG_MAX_LEVELS];      // their level indices
    uint32_t rows[HG_MAX_LEVELS];    // (N_l + 1)^d rows each
    int64_t chunk;                   // points per CTA (grid.x = ceil(n / chunk))
    int32_t smem_bytes;              // dynamic shared memory per CTA
};

struct Tables {
    const void* ptr[5];         // order table k (for the vector path: ptr[0] is the packed row base)
    int64_t ls[5], rs[5];       // level / row strides in elements
};

struct Grads {
    float* ptr[5];
    int64_t ls[5], rs[5];
};

struct FwdParams {
    Common c;
    Tables tab;
    const float* coords;
    float* gamma;
    float* dgamma;
    float* lap;
    float* hess;      // full-Hessian forward only
    float* stencil;   // finite-difference forward only: the 2d stencil encodings
    float eps, half_inv_eps, inv_eps2;  // finite-difference step, 1/(2 eps), 1/eps^2 (fp32)
};

struct BwdParams {
    Common c;
    Priv priv;
    Grads grad;
    const float* coords;
    const float* g_gamma;
    const float* g_dgamma;
    const float* g_lap;
    const float* g_hess;  // full-Hessian backward only
    const float* g_stencil;               // finite-difference backward only
    float eps, half_inv_eps, inv_eps2;    // as FwdParams
};

struct IdxParams {
    Common c;
    const float* coords;
    uint32_t* idx;
};

// Memory-only replay of an encoding launch's row stream (roofline probe).
struct ReplayParams {
    Common c;
    const float* coords;
    char* base;              // packed table (gather) or fp32 gradient table (RED), level 0 row 0
    int64_t level_bytes;     // bytes between levels
    int32_t row_bytes;       // bytes per vertex row
    int32_t lanes;           // lanes sharing a row; each moves row_bytes / lanes bytes
    float* sink;             // gather only: one float per thread
};

// Launchers (one per kernel family); return the cudaError_t of the launch.
// fc: features per pass (1 or 2); vec: whole-row vector access (packed layout).
// hess: the full-Hessian variant (outputs / upstream gradients in hess / g_hess
// instead of lap / g_lap).
int launch_hermite_fwd(const FwdParams& p, int fc, bool vec, int dtype, bool hess, void* stream);
int launch_hermite_bwd(const BwdParams& p, int fc, bool vec, bool hess, void* stream);
int launch_linear_fwd(const FwdParams& p, int fc, bool vec, int dtype, void* stream);
int launch_linear_bwd(const BwdParams& p, int fc, bool vec, void* stream);
int launch_linear_fd_fwd(const FwdParams& p, int fc, bool vec, int dtype, void* stream);
// Gaussian-RBF grid: eps (FwdParams/BwdParams.eps) is the kernel width in grid units, rings 1..4.
int launch_rbf_fwd(const FwdParams& p, int fc, int rings, int dtype, void* stream);
int launch_rbf_bwd(const BwdParams& p, int fc, bool vec, int rings, void* stream);
int launch_linear_fd_bwd(const BwdParams& p, int fc, bool vec, void* stream);
int launch_indices(const IdxParams& p, void* stream);
// red: RED replay (adds 1.0 to every float of each chunk), else gather replay.
int launch_replay(const ReplayParams& p, bool red, void* stream);

// SIREN chain-rule consumer of the encoding.  Rows r of a point: 0 = gamma,
// 1..d = d gamma / d x_i, d + 1 = lap gamma (each feature-major, [K][n]).
struct SirenParams {
    int32_t d, K, H, O;
    int32_t tp;          // threads per point (forward H / 16, backward H / 8: 16 or 8 hidden units each)
    int32_t pts;         // points per tile (CTA threads / tp)
    int32_t nbuf;        // input tile buffers: 2 = the next tile loads while this one computes
    int64_t n;
    float omega;
    const float* in[6];  // rows; NULL = zero
    const float *W1, *b1, *W2, *b2;
    // forward outputs ([O][n], [d][O][n], [O][n]; NULL = not wanted)
    float *u, *du, *lapu;
    // backward: upstream gradients (NULL = zero), input gradients (NULL = not wanted),
    // weight gradients (accumulated; NULL = not wanted)
    const float *g_u, *g_du, *g_lapu;
    float* g_in[6];
    float *gW1, *gb1, *gW2, *gb2;
};
// Dynamic shared memory of one CTA, and the launch (persistent CTAs, at most `ctas`).
// siren_bwd_tiles sets the backward's tp and pts (its CTAs are twice the forward's).
void siren_bwd_tiles(SirenParams& p);
size_t siren_smem_bytes(const SirenParams& p, bool bwd);
int launch_siren_fwd(const SirenParams& p, int ctas, void* stream);
int launch_siren_bwd(const SirenParams& p, int ctas, void* stream);
int siren_ctas_per_sm(const SirenParams& p, bool bwd, int* ctas);
// Fused encoder + SIREN forward (d = 2 or 3, packed F = 2 table of dtype `dtype`,
// one input buffer): CTAs per SM, and the launch of `ctas` persistent CTAs.
int encode_siren_ctas_per_sm(const SirenParams& p, int dtype, int* ctas);
int launch_encode_siren_fwd(const SirenParams& p, const FwdParams& e, int dtype, int ctas, void* stream);
// Tensor-core SIREN forward (split tf32 first layer, 128-point tiles, one CTA per SM): whether a shape
// takes it (d >= 3, H >= 64, (d + 2) H <= 512 TMEM columns, operands within `smem_max` bytes of shared
// memory), and its launch.
bool siren_tc_usable(const SirenParams& p, int smem_max);
int launch_siren_fwd_tc(const SirenParams& p, void* stream);

}  // namespace hg
