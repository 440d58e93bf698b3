/*
 * hm.h -- C ABI of the GB300 update-phase library (libhm).
 *
 * Implements the update phase of "SS-HSDP: Efficient and Flexible Sharded
 * Data Parallelism via Runtime-Update Decoupling" on one GPU:
 *   f0  momentum            (section 3.1 example EG1; Figure 4 "Local momentum")
 *   P2P fragment gather     (section 3.2 "Distributed updates"; section 3.4)
 *   f1  batched Newton-Schulz (EG1; section 4.1 "Batched Update and Transform")
 *   P2P return + f2 update  (EG1; section 3.4; Figure 4 "Local main-weight update")
 *   G   MXFP8 requant       (EG1; Figure 4 "K-major scale layout", "UE8M0")
 * plus the elementwise AdamW update (section 5.2) and the data-tree / shard-
 * chain metadata the update is planned from (section 3.2, section 4.2).
 *
 * The ZeRO ranks are emulated: every field (w, m, g, u, v, q, s) is ONE device
 * allocation holding `so` rank segments in rank order, each starting on a
 * multiple of HM_SEG_ALIGN elements with HM_SEG_GAP canary elements before,
 * between and after them.  The point-to-point exchange of the paper becomes an
 * in-HBM gather / scatter between segments.
 *
 * Conventions for every call:
 *   - Return value: HM_OK (0) or a negative hm_status; hm_status_str() names it.
 *   - Device pointers are caller-owned (e.g. allocated by PyTorch); the
 *     library never frees them.  Handles (hm_tree, hm_chain, hm_muon_plan) are
 *     host metadata owned by the library and released by their *_destroy call.
 *   - Geometry, alignment, overlap and unit checks run on the host before any
 *     launch; a failing check launches nothing and returns its status.
 *   - Launches are asynchronous on the given stream (a cudaStream_t passed as
 *     void*; NULL = the legacy default stream).  A launch error is returned as
 *     HM_ERR_CUDA.  Device-side wait timeouts are recorded in a device error
 *     word that hm_device_error() reads.
 *   - Element offsets and lengths are int64 element counts, not bytes, unless
 *     a name says _bytes.
 */
#ifndef HM_H
#define HM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int hm_status;
#define HM_OK             0
#define HM_ERR_ARG       -1   /* null pointer, bad enum, negative size          */
#define HM_ERR_GEOMETRY  -2   /* view or range outside its parent / list        */
#define HM_ERR_OVERLAP   -3   /* storage overlap where disjointness is required */
#define HM_ERR_ALIGN     -4   /* offset / length not aligned as required        */
#define HM_ERR_DTYPE     -5   /* unsupported dtype for the call                 */
#define HM_ERR_UNITS     -6   /* units do not tile the tensor list              */
#define HM_ERR_CUDA      -7   /* a CUDA runtime / driver call failed            */
#define HM_ERR_ARCH      -8   /* device is not sm_103 (GB300)                   */
#define HM_ERR_TIMEOUT   -9   /* a device-side wait gave up (see hm_device_error) */
#define HM_ERR_WORKSPACE -10  /* workspace too small or not the uploaded one    */
#define HM_ERR_STATE     -11  /* call out of order (e.g. plan not uploaded)     */

typedef enum { HM_U8 = 0, HM_BF16 = 1, HM_F32 = 2, HM_E4M3 = 3 } hm_dtype;

#define HM_SEG_ALIGN 1024   /* elements */
#define HM_SEG_GAP   1024   /* elements */
#define HM_MX_BLOCK  32     /* elements per MXFP8 scale */

/* Name of a status code (static string). */
const char* hm_status_str(hm_status s);

/* Reads and clears the device error word of the current device.  *code = 0
 * when no kernel recorded an error; otherwise the first recorded code (a
 * device-side wait that gave up, HM_ERR_TIMEOUT).  Synchronises the device. */
hm_status hm_device_error(int* code);

/* Number of kernels the calling thread has enqueued through this library
 * since it loaded (every entry point counts each kernel it launches, on any
 * stream).  Host-only: reads a thread-local counter, touches no device.  The
 * difference of two readings around a sequence of calls is the number of
 * kernel launches that sequence made.  The pages define no such call; it
 * exists so that a caller can report how many kernels a step runs. */
hm_status hm_kernel_launches(int64_t* count);

/* ------------------------------------------------------------------------ */
/* Data tree (section 3.2 "Data Tree"): a root node owns one allocation; every
 * other node is a view (parent, byte offset, dtype, shape) and reaches the
 * storage through its accumulated offset. */
typedef struct hm_tree hm_tree;

/* root: device (or host) address of the allocation, NOT owned by the tree;
 * root_bytes > 0.  Node 0 is the root (dtype HM_U8, shape [root_bytes]). */
hm_status create_data_tree(hm_tree** out, void* root, size_t root_bytes);

/* Adds a view of `parent`.  Rejects (HM_ERR_GEOMETRY) a view extending past its
 * parent, (HM_ERR_ALIGN) an accumulated offset not a multiple of the element
 * size, (HM_ERR_ARG) ndim outside 1..8 or a negative extent. */
hm_status data_tree_add_view(hm_tree* t, int parent, size_t byte_off, hm_dtype dtype,
                             int ndim, const int64_t* shape, int* node_out);

/* Address (root + accumulated offset) and accumulated offset of a node. */
hm_status data_tree_resolve(const hm_tree* t, int node, void** ptr, size_t* root_off);

/* HM_ERR_OVERLAP if any two of the given nodes share a byte, else HM_OK. */
hm_status data_tree_check_disjoint(const hm_tree* t, const int* nodes, int n);

void tree_destroy(hm_tree* t);

/* ------------------------------------------------------------------------ */
/* Shard chain (section 3.2 "Shard Chain"; section 4.2 "Fully Zero Copy").
 * A tensor list of n elements is cut at ZeRO-1 edges E_0..E_so (default
 * E_c = 32*floor(c*n/(32*so)); n must be a multiple of 32).  z1 chunk
 * c = i*(so/sw) + j is owned by rank i + j*sw (owners [0,2,1,3] for so = 4,
 * sw = 2).  A level of degree s (sw for z3, sg for z2) has chunk k = z1 chunks
 * [k*so/s, (k+1)*so/s).  Degrees must nest: sw | sg | so. */
typedef struct hm_chain hm_chain;

typedef struct {
    int32_t chunk;        /* chunk index at the requested level            */
    int32_t rank;         /* z1: owning rank; z2/z3: lowest rank holding it */
    int64_t seg_offset;   /* element offset inside that chunk              */
    int64_t unit_offset;  /* element offset inside the queried range       */
    int64_t length;       /* elements                                      */
    int64_t root_offset;  /* z1 only: element offset in the emulated root  */
} hm_fragment;

/* z1_edges: NULL for the default edges, else so+1 non-decreasing multiples of
 * 32 from 0 to n.  edge_shift (only with z1_edges == NULL): NULL, or so+1
 * multiples of 32 added to the default edges (ragged edges; entries 0 and so
 * must be 0).  Rejects unaligned edges or shifts (HM_ERR_ALIGN), edges that
 * decrease or miss 0 / n (HM_ERR_GEOMETRY), degrees that do not nest
 * (HM_ERR_GEOMETRY), n not a multiple of 32 (HM_ERR_ALIGN). */
hm_status shard_chain(hm_chain** out, int64_t n, int so, int sw, int sg, const int64_t* z1_edges,
                      const int64_t* edge_shift);

/* Emulated root layout: *total = elements of one field allocation; bases[r]
 * (so entries, may be NULL) = element offset of rank r's segment; lens[r] =
 * its length; chunk_of_rank[r] = its z1 chunk. */
hm_status shard_chain_layout(const hm_chain* c, int64_t* total, int64_t* bases, int64_t* lens,
                             int32_t* chunk_of_rank);

/* Fragments of the logical range [a, b) at level 1 (z1), 2 (z2) or 3 (z3), in
 * range order.  Writes min(cap, count) entries, *n = count. */
hm_status shard_chain_fragments(const hm_chain* c, int64_t a, int64_t b, int level,
                                hm_fragment* out, int cap, int* n);

/* Adds one view per rank segment (dtype, shape [len_r]) as children of node 0
 * of a field's data tree whose root holds the emulated layout; node ids are
 * written to nodes_out[so]. */
hm_status shard_chain_segment_views(const hm_chain* c, hm_tree* t, hm_dtype dtype, int* nodes_out);

void chain_destroy(hm_chain* c);

/* ------------------------------------------------------------------------ */
/* Muon update of a tensor list (EG1; section 3.4 "Update"; section 4.1). */
typedef struct {
    int64_t offset;   /* element offset of the unit in the tensor list   */
    int32_t rows;     /* a unit is a contiguous rows x cols row-major block */
    int32_t cols;
} hm_unit_desc;

typedef struct hm_muon_plan hm_muon_plan;

/* Plans the update of the units (sorted, disjoint, tiling [0, n) exactly:
 * else HM_ERR_UNITS; rows*cols a multiple of 32: else HM_ERR_ALIGN; rows and
 * cols at most 2^20 and at most 65535 units per shape class: else
 * HM_ERR_GEOMETRY).  Classifies each unit as local (one z1
 * fragment) or straddling, picks its execution rank (owner of its first
 * element), groups units by Newton-Schulz shape class (min, max of rows,
 * cols) and lays out the workspace.  Host only. */
hm_status muon_plan(hm_muon_plan** out, const hm_chain* chain, const hm_unit_desc* units, int n_units);

typedef struct {
    int32_t n_units, n_local, n_straddling, n_classes;
    int64_t staging_elems;    /* elements of the u / v staging of straddling units */
    int64_t workspace_bytes;  /* device workspace muon_update_units needs      */
    int32_t n_fragments;      /* z1 fragments of straddling units               */
} hm_muon_plan_info;
hm_status muon_plan_query(const hm_muon_plan* p, hm_muon_plan_info* info);

/* Per-unit plan facts: *exec_rank, *n_frags, *cls (shape class), *local. */
hm_status muon_plan_unit(const hm_muon_plan* p, int unit, int32_t* exec_rank, int32_t* n_frags,
                         int32_t* cls, int32_t* local);

/* Copies the plan's device tables into `workspace` (device, >= workspace_bytes,
 * 1024-byte aligned) and encodes the tensor maps of its scratch regions.  Must
 * precede muon_update_units with that workspace; calling it again with another
 * workspace re-targets the plan.  Needs a current sm_103 device. */
hm_status muon_plan_upload(hm_muon_plan* p, void* workspace, size_t workspace_bytes, void* stream);

typedef struct {
    float lr;            /* 0.02 */
    float momentum;      /* mu, 0.95 */
    float weight_decay;  /* decoupled, applied in f2 when != 0 */
    float eps;           /* Newton-Schulz normalisation, 1e-7 */
    float ns_a, ns_b, ns_c;   /* 3.4445, -4.7750, 2.0315 */
    int32_t ns_steps;    /* 5 */
    int32_t nesterov;    /* 0: u = bf16(m); 1: u = bf16(g + mu*m) */
    int32_t alpha_mode;  /* 0: 1; 1: sqrt(max(1, rows/cols)); 2: 0.2*sqrt(max(rows, cols)) */
} hm_muon_hparams;

typedef struct {  /* device roots, each in the chain's emulated layout */
    float*    w;   /* fp32 main weight,     total elements         */
    float*    m;   /* fp32 momentum                                  */
    const float* g;/* fp32 main gradient                             */
    uint16_t* u;   /* bf16 intermediate u (bit patterns)             */
    float*    v;   /* fp32 update direction v                        */
    uint8_t*  q;   /* E4M3 runtime weight, same element offsets as w */
    uint8_t*  s;   /* UE8M0 scales, element offset / 32              */
} hm_muon_bufs;

#define HM_STAGE_F0      1   /* m <- mu m + g; u = bf16(m)                 */
#define HM_STAGE_GATHER  2   /* u fragments of straddling units -> staging  */
#define HM_STAGE_NS      4   /* f1 for every unit -> v                      */
#define HM_STAGE_F2      8   /* v fragments -> owners; w <- w - lr alpha v  */
#define HM_STAGE_REQUANT 16  /* G: w -> (q, s) in every segment             */
#define HM_STAGE_ALL     31
/* Fused update (SS-HSDP section 4.2 "Fully Zero Copy": no extra copies):
 * with HM_STAGE_FUSED, F0 and GATHER run as one pass (f0 also writes the u
 * fragments of straddling units into their staging, so u is read once), and
 * F2 and REQUANT run as one pass (w is read once; its new value is quantized
 * as it is written).  F0 and GATHER must be requested together, and F2 and
 * REQUANT together (else HM_ERR_ARG); NS runs as usual.  Outputs m, u, v, w,
 * q, s equal those of the unfused stages bit for bit. */
#define HM_STAGE_FUSED   32
#define HM_STAGE_ALL_FUSED 63
/* u and v as scratch (section 3.1, EG1: both are update-scoped intermediates,
 * u consumed by f1 and v by f2).  HM_STAGE_SCRATCH requires HM_STAGE_FUSED,
 * and NS only together with F2 and REQUANT (else HM_ERR_ARG).  With F0, u is
 * not written anywhere: f0 runs inside the pass that lays out each shape
 * class's Newton-Schulz input X0 = u in the workspace (with the norm's partial
 * sums and the unit scales), reading g and m -- and writing m -- in the rank
 * segments that hold them, so the fragment gather needs no pass either; the
 * next NS stage on this plan (with or without SCRATCH) starts from that input
 * instead of preparing it from the u root.  An F0 stage without SCRATCH, or
 * muon_plan_upload, drops the prepared input.  With NS, the last Newton-Schulz product of every
 * unit whose cols and fragments are multiples of HM_MX_BLOCK applies f2 and G
 * to that unit in its epilogue, reading w and writing w, q and s directly, and
 * stores no v for it (v keeps its previous contents); the fused F2 + REQUANT
 * pass then covers only the other units (a call with F2 and REQUANT but without
 * NS runs the pass over every unit, from v).  m, v (where written), w, q and s
 * equal those of HM_STAGE_ALL_FUSED bit for bit.  HM_STAGE_STEP is the whole
 * update phase in this fastest form; it may also be split into
 * F0 | GATHER | FUSED | SCRATCH and NS | F2 | REQUANT | FUSED | SCRATCH. */
#define HM_STAGE_SCRATCH 64
#define HM_STAGE_STEP    127

/* Runs the selected stages, in the order above, on `stream`.  u and v of
 * straddling units live in the workspace staging; v of local units is
 * written to the v root at the unit's own offsets.  A plan serves one stream
 * at a time: calls on one plan must not run concurrently (they share the
 * workspace and the plan's cached per-unit steps).
 * Allocates nothing and launches only kernels on `stream`, so a call can be
 * captured into a CUDA graph and replayed, provided one call with the same
 * lr and alpha_mode ran outside the capture first: a change of either
 * re-uploads the per-unit step table from host memory (a copy a capture
 * cannot hold).  Replays read that table (and the per-unit steps of the
 * last products) from the workspace, so a later uncaptured call with a new
 * lr also updates the graph's steps; the other scalars -- mu, the weight
 * decay factor fp32(1 - lr * wd), eps, a, b, c -- are kernel arguments fixed
 * at capture. */
hm_status muon_update_units(const hm_muon_plan* p, const hm_muon_bufs* bufs,
                            const hm_muon_hparams* hp, void* workspace, size_t workspace_bytes,
                            int stages, void* stream);

/* Device address of a straddling unit's u / v staging (after upload). */
hm_status muon_plan_staging(const hm_muon_plan* p, int unit, uint16_t** u_stage, float** v_stage);

void muon_plan_destroy(hm_muon_plan* p);

/* ------------------------------------------------------------------------ */
/* Fused elementwise AdamW over one flat shard (section 5.2; PyTorch AdamW
 * semantics: decoupled weight decay, bias correction with step t >= 1).
 * w, m, v: fp32 [n]; g: [n] of g_dtype (HM_BF16 or HM_F32).  n = 0 is a no-op.
 * Pointers must be 16-byte aligned (HM_ERR_ALIGN). */
typedef struct {
    float lr, beta1, beta2, eps, weight_decay;
    int32_t step;
} hm_adamw_hparams;

hm_status adamw_update_flat(float* w, const void* g, hm_dtype g_dtype, float* m, float* v,
                            int64_t n, const hm_adamw_hparams* hp, void* stream);

/* ------------------------------------------------------------------------ */
/* G: MXFP8 requantization (EG1; OCP MX format): for every 1 x 32 block along K
 * of each [rows][K] fp32 tensor, e = clamp(floor(log2 amax) - 8, -127, 127),
 * scale code e + 127, elements E4M3 = RNE(x * 2^-e) saturated to +-448.
 * Codes are written at dst_offset (same [rows][K] layout: the packed QKV /
 * grouped-GEMM layout of the source), scales as [rows][K/32] at
 * scale_offset.  K must be a multiple of 32; src_offset and dst_offset
 * multiples of 32 (HM_ERR_ALIGN).  n = 0 is a no-op. */
typedef struct {
    int64_t src_offset;    /* elements of w     */
    int64_t dst_offset;    /* elements of q     */
    int64_t scale_offset;  /* elements of s     */
    int64_t rows;
    int64_t k;
} hm_mx_tensor;

hm_status mxfp8_requant_packed(const float* w, uint8_t* q, uint8_t* scales,
                               const hm_mx_tensor* tensors, int n, void* stream);

/* ------------------------------------------------------------------------ */
/* Newton-Schulz of one unit without any device allocation.  The paper has no
 * counterpart: this entry point exists for callers that cannot call
 * cudaMalloc -- code inside a framework whose caching allocator already owns
 * all device memory (a cudaMalloc of its own would fail or fragment the
 * pool), and latency-critical paths that must not take the driver's
 * allocation lock or risk the implicit synchronisation an allocation brings.
 *
 * u: device, rows x cols bf16 bit patterns, row-major, 16-byte aligned; v:
 * device, rows x cols fp32 output, row-major; both caller-owned.  Computes
 * what the Newton-Schulz stage of muon_update_units computes for one unit
 * (same kernels): X0 = u / (||u||_F + eps), transposed when rows > cols,
 * hp->ns_steps iterations of X = aX + (bA + cA^2)X with A = X X^T, v = X.
 *
 * Every intermediate lives in one file-scope __device__ array of
 * HM_NOALLOC_SCRATCH_BYTES bytes that each GPU loading the library holds
 * until the process exits.  Limits: min(rows, cols) <= HM_NOALLOC_MAX_MIN_DIM
 * and max(rows, cols) <= HM_NOALLOC_MAX_MAX_DIM, else HM_ERR_WORKSPACE;
 * rows*cols a multiple of 8 and the alignments above, else HM_ERR_ALIGN.
 * The first call on a device looks up the array's device address (once per
 * device, with that device current); make that first call before any stream
 * capture.  All calls on a device share the array and it keeps the last
 * call's contents (every call overwrites what it reads), so calls that
 * overlap on the GPU -- on different streams, or concurrent host threads --
 * race; serialise them.  Launches on `stream`; allocates nothing. */
#define HM_NOALLOC_MAX_MIN_DIM 128
#define HM_NOALLOC_MAX_MAX_DIM 8192
#define HM_NOALLOC_SCRATCH_BYTES 4197376
hm_status newton_schulz_noalloc(const uint16_t* u, int32_t rows, int32_t cols, float* v,
                                const hm_muon_hparams* hp, void* stream);

/* ------------------------------------------------------------------------ */
/* G with 32 x 32 blocks (section 3.1 EG1: "32 x 32 block quantization in a
 * k-major layout"): one UE8M0 scale per 32-row x 32-column block of each
 * [rows][K] tensor, e = clamp(floor(log2 amax) - 8, -127, 127) over the 1024
 * elements, elements E4M3 RNE saturated.  A block spans 32 rows, so it can
 * straddle ZeRO-1 edges: with a chain, w and q are emulated roots in the
 * chain's layout and every block row is read from (and written to) the rank
 * segment that holds it -- the in-HBM form of gathering the block to an
 * execution rank.  chain == NULL: w and q are flat, logical order.
 * tensors[i]: src_offset = logical element offset of the tensor (a multiple
 * of 32), rows and k multiples of 32 (else HM_ERR_ALIGN), scale_offset = byte
 * offset of its [rows/32][k/32] scale matrix in `scales`; dst_offset is not
 * used (codes land at each element's own position in q).  At most 256 ranks
 * (HM_ERR_ARG).  n = 0 is a no-op. */
hm_status mxfp8_requant_32x32(const hm_chain* chain, const float* w, uint8_t* q, uint8_t* scales,
                              const hm_mx_tensor* tensors, int n, void* stream);

/* Tw's scale relayout (EG1: scales are relaid out for the GEMM kernel;
 * section 4.1: batched across tensors).  Each item takes a K-major scale
 * matrix [rows / block_rows][kb] (block_rows 1 for 1 x 32 blocks, 32 for
 * 32 x 32 blocks, whose scale is repeated over its 32 rows) at src + src_offset
 * and writes the 128 x 4 tiled layout read by block-scaled tensor-core GEMMs
 * (the cuBLAS "1D block scaling factors" layout) at dst + dst_offset:
 * ceil(rows/128) * ceil(kb/4) tiles of 512 bytes, tile (i, j) at
 * (i * ceil(kb/4) + j) * 512, row r / column c of a tile at
 * (r % 32) * 16 + (r / 32) * 4 + c, padding zero.  rows % block_rows == 0
 * (HM_ERR_ALIGN).  n = 0 is a no-op. */
typedef struct {
    int64_t src_offset;   /* bytes */
    int64_t dst_offset;   /* bytes */
    int64_t rows;         /* weight rows */
    int64_t kb;           /* scales per row = K / 32 */
    int32_t block_rows;   /* 1 or 32 */
    int32_t pad;
} hm_scale_relayout;

hm_status mxfp8_scale_relayout(const uint8_t* src, uint8_t* dst, const hm_scale_relayout* items, int n,
                               void* stream);

/* ------------------------------------------------------------------------ */
/* Outer reduce-scatter of the main gradient, emulated in HBM (section 3.4
 * Update: Tg maps the accumulated gradients to the update representation and
 * the outer reduce-scatter produces the ZeRO-1 main-gradient shards; section
 * 4.3 ZeroSM reduce-scatter: intra-node FP32 reduce, inter-node exchange,
 * final FP32 reduce accumulating into the persistent gradient; node-local
 * partials optionally BF16 with stochastic rounding; Table 4: the SR seed /
 * counter state is restored on the same logical rank).
 *
 * parts: device, n_parts x n fp32, row p = contribution of rank p in logical
 * order (n = the chain's tensor-list length); ranks form nodes of
 * ranks_per_node consecutive rows.  g: device root in the chain's layout.
 * For every element i (written in the rank segment that owns it):
 *   s_k   = fp32 sum of the node's rows, in row order
 *   p_k   = s_k (HM_RS_FP32) | bf16_RNE(s_k) (HM_RS_BF16) |
 *           bf16_SR(s_k) (HM_RS_BF16_SR: 16 random bits added to the low half
 *           of the fp32 pattern, then truncated; bits = 16-bit field (i mod 8)
 *           of the 128-bit Philox4x32-10 output for counter (i/8 mod 2^32,
 *           i/8 div 2^32, k, offset mod 2^32) and key (seed mod 2^32, seed div
 *           2^32); field f = bits 16*(f mod 2).. of word f/2)
 *   total = fp32 sum of the p_k in node order
 *   g     = accumulate ? g + total : total
 * Rejects n_parts not a multiple of ranks_per_node (HM_ERR_GEOMETRY), a bad
 * mode (HM_ERR_ARG), pointers not 16-byte aligned (HM_ERR_ALIGN). */
#define HM_RS_FP32    0
#define HM_RS_BF16    1
#define HM_RS_BF16_SR 2
hm_status reduce_scatter_grad(const hm_chain* chain, const float* parts, int n_parts, int ranks_per_node,
                              float* g, int mode, int accumulate, uint64_t seed, uint64_t offset, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* HM_H */
