// Internal declarations shared by the host planner (hm_host.cpp) and the
// CUDA kernels (hm_elementwise.cu, hm_ns.cu).  Not part of the C ABI.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda.h>
#include <cuda_runtime.h>

namespace hm {

// Device-side error codes recorded in the library's device error word.
constexpr int kDevErrTimeout = -9;   // == HM_ERR_TIMEOUT

// One entry of a range table: the same element index d in [0, len) maps to
// element a + d of one buffer, b + d of another and, for MXFP8 scales,
// (c + d) / 32 of a third.  `prefix` is the exclusive prefix sum of len over
// the table, so a table describes one virtual index space [0, total).
struct Range {
    int64_t a;
    int64_t b;
    int64_t c;
    int64_t len;
    int64_t prefix;
    float   step;   // f2: fp32(lr * alpha) of the unit the range belongs to
    int32_t flags;  // f2: bit 0 = v read from the workspace staging;
                    // f0: bit 1 = also write u to the staging at b + d
};
static_assert(sizeof(Range) == 48, "Range layout");

constexpr int kInlineRanges = 32;

// Kernel argument: a table either in device memory (tab != nullptr) or
// inline in the kernel's parameter space.
struct RangeArgs {
    const Range* tab;
    int32_t n;
    int32_t pad;
    int64_t total;
    Range inl[kInlineRanges];
};

// One Newton-Schulz unit.
struct NsUnit {
    int64_t u_off;   // element offset of u in the u root or the u staging
    int64_t v_off;   // element offset of v in the v root or the v staging
    int32_t rows;    // unit as stored: rows x cols, row-major
    int32_t cols;
    int32_t flags;   // kNs* bits
    float   step;    // kNsEpiUpdate: fp32(lr * alpha), as in the f2 table
    int32_t frag0;   // first of the unit's nfrag entries in the fragment table (unit order)
    int32_t nfrag;
};
static_assert(sizeof(NsUnit) == 40, "NsUnit layout");
constexpr int kNsUStaged = 1;       // u read from staging
constexpr int kNsVStaged = 2;       // v written to staging
constexpr int kNsTransposed = 4;    // rows > cols: X = u^T
constexpr int kNsEpiUpdate = 8;     // the last product may apply f2 and G itself: cols and
                                    // every fragment a multiple of 32, so each 1 x 32 MX
                                    // block is one row piece of the unit in one fragment

// Where a unit's elements live in the roots of w, q (element offsets) and s
// (offset / 32): unit elements [unit_off, next entry's unit_off) start at
// root_off.  A unit's entries are in unit order; a local unit has one.
struct NsFrag {
    int64_t unit_off;
    int64_t root_off;
};

// A Newton-Schulz shape class: units with the same (m, n) = (min, max) of
// (rows, cols).  X is stored padded to mp x np (mp multiple of 128, np
// multiple of 64) with zeros outside m x n; the zero padding stays zero
// through every iteration.
struct NsClassDev {
    int32_t m, n, mp, np;
    int32_t n_units;
    int32_t first_unit;  // into the NsUnit table
    int32_t parts;       // norm partial sums per unit: one per 64 x 64 tile of X
    size_t x_off[2], a_off, b_off, part_off, inv_off;  // workspace bytes
    int32_t sym_tiles;   // tiles of the mp x mp output on or above the diagonal
    size_t sym_off;      // workspace bytes: their (tm << 16 | tn) list, L2-friendly order
    int32_t pair_tiles;  // the same for the 256 x 256 tiles of the CTA-pair kernel
    size_t pair_off;
};

// Epilogue kinds of the Newton-Schulz GEMM.
enum GemmEpi : int {
    kEpiGram = 0,    // out = bf16(acc)                         (A = X X^T)
    kEpiPoly = 1,    // out = bf16(alpha*acc + beta*add)        (B = b A + c A A)
    kEpiUpdate = 2,  // out = bf16(acc + beta*add)               (X = a X + B X)
    kEpiFinal = 3,   // v   = fp32(acc + beta*add), per-unit destination
};

struct GemmParams {
    int32_t M, N, K;            // per unit; M multiple of 128, N multiple of 32
    int32_t units, tiles_m, tiles_n, num_kb;
    int32_t epi;
    float alpha, beta;
    uint16_t* out;       int64_t out_us;   int32_t ld_out;   // [units][M][N]
    const uint16_t* add; int64_t add_us;   int32_t ld_add;   // [units][M][N]
    const NsUnit* ns_units;                                   // final: destinations
    float* v_root;
    float* v_stage;
    int32_t m_real, n_real;
    int32_t* err;
    const int32_t* tile_tab;  // optional tile list per unit ((tm << 16) | tn); nullptr = full grid
    int32_t tab_len;
    int32_t sym;              // symmetric output: write (i, j) and (j, i) for j >= i only
    int32_t group_m;          // tile-rows per raster band of the full grid (0 = 8)
    int32_t inject_no_ready;  // failure test: never signal an accumulator as ready
    int32_t* pace;            // CTA-pair kernel: 2 device ints (tiles issued, pairs done), zero between
                              // launches; nullptr = pairs run unpaced
    const float* unit_scale;  // first iteration: s = 1 / (||u|| + eps) per unit, X0 being u itself:
                              // the Gram output is scaled by s^2, the B X output (acc + beta*add) by s;
                              // nullptr = none
    // final product with the update folded in (units flagged kNsEpiUpdate):
    // w <- w*decay - step*v and G on the new w, v itself never stored
    int32_t fuse_update;
    int32_t has_decay;
    float decay;
    const NsFrag* frags;
    float* w;
    uint8_t* q;
    uint8_t* s;
};

// Whole Newton-Schulz of a class whose Gram size mp is 128 in one persistent
// kernel (every product of every iteration; X read once and written once per
// iteration).  g carries the last product's epilogue fields (ns_units,
// v_root, v_stage, m_real, n_real, fuse_update and its w, q, s, frags, decay),
// err, inject_no_ready and unit_scale (1 / (||u|| + eps) per unit).
struct SmallNsParams {
    GemmParams g;
    int32_t units;    // units of the class
    int32_t u0;       // first unit this launch takes (units u0 .. units - 1; launch_ns_small sets it)
    int32_t np;       // padded row length of X (multiple of 64)
    int32_t steps;    // Newton-Schulz iterations
    int32_t reverse;  // alternate the tile order of consecutive passes over X
    float a, b, c;
};

// chain geometry the device needs: z1 edges and the segment base of every chunk
constexpr int kMaxChainRanks = 256;
struct ChainArgs {
    int32_t so;          // 0: flat, logical == root
    int32_t pad;
    int64_t edges[kMaxChainRanks + 1];
    int64_t chunk_base[kMaxChainRanks];
};

constexpr int kMaxMx32Tensors = 32;
struct Mx32Args {
    int32_t n;
    int32_t pad;
    int64_t block_prefix[kMaxMx32Tensors + 1];  // exclusive prefix of 32-row x 128-column strip counts
    int64_t src[kMaxMx32Tensors];
    int64_t k[kMaxMx32Tensors];
    int64_t scale_off[kMaxMx32Tensors];
};

constexpr int kMaxRelayoutItems = 32;
struct RelayoutArgs {
    int32_t n;
    int32_t pad;
    int64_t work_prefix[kMaxRelayoutItems + 1];  // exclusive prefix of 128-row x 160-column work units
    int64_t src[kMaxRelayoutItems];
    int64_t dst[kMaxRelayoutItems];
    int64_t rows[kMaxRelayoutItems];
    int64_t kb[kMaxRelayoutItems];
    int32_t block_rows[kMaxRelayoutItems];
    int32_t flags[kMaxRelayoutItems];  // kRelayout* bits
};
constexpr int kRelayoutSrc16 = 1;     // src + src offset and kb are multiples of 16: 16-byte row loads
constexpr int kRelayoutDst16 = 2;     // dst + dst offset is 16-byte aligned: one 16-byte store per group

// ---- launchers (return cudaGetLastError() of the launch) -----------------
// Kernels launched by the calling thread through the library (every launch
// site calls note_launch once per kernel it enqueues).
void note_launch();
int64_t launches_issued();
int device_sm_count();

// Grid of a grid-stride kernel: every CTA resident at once (SM count x the
// CTAs per SM that the kernel's registers, shared memory and block size
// allow), or one CTA per work item when there are fewer.  A larger grid
// would leave its last CTAs to run alone after the others have finished.
template <class Kernel>
inline int resident_grid(Kernel kernel, int threads, int64_t items) {
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, 0) != cudaSuccess || per_sm < 1)
        per_sm = 1;
    const int64_t cap = static_cast<int64_t>(device_sm_count()) * per_sm;
    if (items < 1) items = 1;
    return static_cast<int>(items < cap ? items : cap);
}
int32_t* device_error_word();

// stage_only: ranges flagged for the staging write u there only (not in the u root)
cudaError_t launch_f0(const RangeArgs& ra, float* m, const float* g, uint16_t* u, uint16_t* u_stage,
                      float mu, int nesterov, int stage_only, cudaStream_t st);
cudaError_t launch_copy_bf16(const RangeArgs& ra, const uint16_t* src, uint16_t* dst, cudaStream_t st);
cudaError_t launch_f2(const RangeArgs& ra, float* w, const float* v_root, const float* v_stage,
                      float decay, int has_decay, cudaStream_t st);
cudaError_t launch_requant(const RangeArgs& ra, const float* w, uint8_t* q, uint8_t* s, cudaStream_t st);
cudaError_t launch_f2_requant(const RangeArgs& ra, float* w, const float* v_root, const float* v_stage,
                              uint8_t* q, uint8_t* s, float decay, int has_decay, cudaStream_t st);
cudaError_t launch_adamw(float* w, const void* g, int g_bf16, float* m, float* v, int64_t n,
                         float lr, float beta1, float beta2, float eps, float decay,
                         float step_size, float inv_sqrt_bc2, cudaStream_t st);

cudaError_t launch_requant_32x32(const ChainArgs& ch, const Mx32Args& ta, const float* w, uint8_t* q,
                                 uint8_t* scales, cudaStream_t st);
cudaError_t launch_scale_relayout(const RelayoutArgs& ra, const uint8_t* src, uint8_t* dst, cudaStream_t st);

struct RsArgs {
    const float* parts;
    int64_t stride;      // elements per contribution row (= n)
    int32_t n_parts, ranks_per_node, mode, accumulate;
    uint32_t seed_lo, seed_hi, offset_lo, pad;
};
cudaError_t launch_reduce_scatter(const RangeArgs& ra, const RsArgs& a, float* g, cudaStream_t st);

// X0 (u itself, laid out and padded) and the per-tile sums of squares of u;
// then 1 / (||u|| + eps) per unit from those sums
cudaError_t launch_ns_prepare(const NsClassDev& c, const NsUnit* units_dev, const uint16_t* u_root,
                              const uint16_t* u_stage, char* ws, cudaStream_t st);
cudaError_t launch_ns_norm(const NsClassDev& c, char* ws, float eps, cudaStream_t st);
// f0 of every element of the class's units (m updated where it lives in the
// rank segments) with u going straight into X0 and the norm's partial sums:
// the prepare pass without a stored u (frags: every unit's fragment table)
cudaError_t launch_ns_f0_prepare(const NsClassDev& c, const NsUnit* units_dev, const NsFrag* frags_dev, float* m,
                                 const float* g, float mu, int nesterov, char* ws, cudaStream_t st);
// b_mn: the B operand is MN-major (its map has 64 x 64 boxes, N innermost)
cudaError_t launch_ns_gemm(const CUtensorMap& tma, const CUtensorMap& tmb, const GemmParams& p,
                           int bn, int b_mn, cudaStream_t st);
// The whole Newton-Schulz of a class with mp = 128, after the prepare pass and
// the norm: x0 and x1 map the two X buffers [units][128][np] with 128-row x
// 64-column boxes; X0 is in buffer 0.
cudaError_t launch_ns_small(const CUtensorMap& x0, const CUtensorMap& x1, const SmallNsParams& p, cudaStream_t st);
// CTA-pair (cta_group::2) variant: 256 x 256 tiles, M a multiple of 128; both
// operand maps use 128-row boxes (64 x 64 boxes for an MN-major B)
cudaError_t launch_ns_gemm_pair(const CUtensorMap& tma, const CUtensorMap& tmb, const GemmParams& p, int b_mn,
                                cudaStream_t st);

}  // namespace hm
