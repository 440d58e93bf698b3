// f1: batched Newton-Schulz on sm_103a tensor cores.
//
// SS-HSDP section 3.1 (example EG1: f1 applies Newton-Schulz to the complete
// BF16 intermediate u and writes the FP32 direction v to separate scratch) and
// section 4.1 (f1 groups matrices with matching shapes for batched GEMMs).
// Per unit (rows x cols, m = min, n = max):
//   X0 = u / (||u||_F + eps), taken as u^T when rows > cols (m x n);
//   repeat: A = X X^T;  B = b A + c A A;  X = a X + B X;
//   v = X (transposed back).
// A, B and X are rounded to bf16 after each product (fp32 accumulation in
// TMEM); the last product is written to v in fp32 or, when the caller folds
// f2 and G into it, applied to w and quantized to (q, s) without storing v.
// X0 is stored as u itself (exact in bf16) and s = 1 / (||u||_F + eps) enters
// the first iteration's epilogues: A = s^2 (u u^T), X1 = s (a u + B u) -- the
// same products with the scale applied in fp32 after the sum instead of
// rounding s u to bf16 first.
//
// Layout in the workspace, per shape class of U units:
//   X[2]   bf16 [U][mp][np]   (ping-pong)
//   A, B   bf16 [U][mp][mp]
// with mp = m rounded up to 128 and np = n rounded up to 64; the padding is
// zero and stays zero.  A = X X^T contracts rows of X with rows of X and A A
// rows of A with rows of A (A is symmetric): both operands K-major.  B X
// contracts rows of B with columns of X: B is K-major, X is read as an
// MN-major operand (N contiguous), so X^T is never stored.
//
// GEMM kernels: persistent, 320 threads per CTA.  ns_gemm_kernel runs one
// CTA per SM on 128-row tiles; ns_gemm_pair_kernel (further down) runs CTA
// pairs on 256 x 256 tiles with the same roles.  Single CTA:
//   warp 0      TMA producer: a 128x64 A box and a BNx64 K-major B box (or
//               BN/64 boxes of 64 N x 64 K for an MN-major B), 128-byte
//               swizzle, STAGES-deep mbarrier ring;
//   warp 1      allocates TMEM and issues tcgen05.mma (M=128, N=BN, K=16)
//               from one lane into a double-buffered fp32 accumulator;
//   warps 2-9   epilogue, two warps per TMEM lane quadrant, each draining
//               half of the tile's columns: tcgen05.ld 32x32b rows out of
//               TMEM, fused element-wise tail, global stores.
// Every mbarrier wait is bounded (2 s of %globaltimer); on timeout the CTA
// records HM_ERR_TIMEOUT in the device error word, lets every role finish,
// waits for its own TMA copies and MMAs, frees TMEM and returns.
#include "hm_internal.h"
#include "hm_mx_device.cuh"

#include <cuda_bf16.h>

namespace hm {

namespace {

// ---------------------------------------------------------------------------
// Frobenius norm: the prepare pass below leaves one sum of squares of u per
// 64 x 64 tile of X; this kernel adds a unit's tiles in a fixed order and
// writes 1 / (sqrt + eps).
// ---------------------------------------------------------------------------
constexpr int kNormThreads = 256;

__global__ void __launch_bounds__(kNormThreads) ns_norm_final_kernel(const float* __restrict__ partials, int parts,
                                                                     float* __restrict__ inv, float eps) {
    // one CTA per unit: thread t adds tiles t, t + 256, .., then a shuffle tree
    // per warp and the 8 warp sums in order -- the same order on every call
    __shared__ float red[kNormThreads / 32];
    const int unit = blockIdx.x;
    const float* pu = partials + static_cast<int64_t>(unit) * parts;
    float s = 0.f;
    for (int k = threadIdx.x; k < parts; k += kNormThreads) s += pu[k];
#pragma unroll
    for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = s;
    __syncthreads();
    if (threadIdx.x == 0) {
        float tot = 0.f;
#pragma unroll
        for (int k = 0; k < kNormThreads / 32; ++k) tot += red[k];
        inv[unit] = 1.0f / (sqrtf(tot) + eps);
    }
}

// ---------------------------------------------------------------------------
// X0 from u: 64x64 tiles of X coordinates through shared memory.  Both the
// read of u (in either orientation) and the write of X move 16-byte vectors
// of 8 bf16 when the row length allows it (n, resp. m, a multiple of 8).
// X0 is u itself (bf16, exact): the factor 1 / (||u|| + eps) enters the first
// iteration's products instead (X X^T times its square, B X times it), so the
// pass also leaves the tile's sum of squares of u, the norm's partial sum, and
// u is read once.
// ---------------------------------------------------------------------------
constexpr int kPrepThreads = 128;  // 4 of the tile's 512 16-byte chunks per thread, loads first

__global__ void __launch_bounds__(kPrepThreads) ns_prepare_kernel(const NsUnit* __restrict__ units,
                                                                   const uint16_t* __restrict__ u_root,
                                                                   const uint16_t* __restrict__ u_stage,
                                                                   float* __restrict__ partials,
                                                                   uint16_t* __restrict__ X, int m, int n, int np) {
    // X orientation.  The 8-element chunk c of row r sits at chunk c ^ (r / 8):
    // the transposed path writes down a column, and without the swizzle the 8
    // rows r, r + 8, .. its lanes hit would share one bank
    __shared__ __align__(16) uint16_t T[64][64];
    __shared__ float red[kPrepThreads / 32];
    auto tx = [](int r, int c) { return ((((c >> 3) ^ (r >> 3)) & 7) << 3) | (c & 7); };
    const int unit = blockIdx.z;
    const NsUnit nu = units[unit];
    const uint16_t* src = ((nu.flags & kNsUStaged) ? u_stage : u_root) + nu.u_off;
    const bool tr = nu.flags & kNsTransposed;
    const int i0 = blockIdx.y * 64, j0 = blockIdx.x * 64;
    // u row r has length ld and 64 consecutive X entries of one tile row map to
    // 64 consecutive u entries of one u row (non-transposed) or of one u column
    const int ld = tr ? m : n;
    const bool vec_ok = (ld & 7) == 0;
    const int rlim = tr ? n : m, clim = tr ? m : n;
    uint4 raw[4];  // 8 bf16 of u per chunk, zero outside the unit
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        const int v = threadIdx.x + t * kPrepThreads;
        const int a = v >> 3, b0 = (v & 7) * 8;  // u-tile row a, 8 entries from b0
        // non-transposed: u row i0+a, cols j0+b0..; transposed: u row j0+a, cols i0+b0..
        const int ur = (tr ? j0 : i0) + a, uc = (tr ? i0 : j0) + b0;
        if (ur < rlim && vec_ok && uc + 8 <= clim) {
            raw[t] = __ldg(reinterpret_cast<const uint4*>(src + static_cast<int64_t>(ur) * ld + uc));
        } else {
            uint32_t h[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) h[k] = (ur < rlim && uc + k < clim) ? src[static_cast<int64_t>(ur) * ld + uc + k] : 0u;
            raw[t] = make_uint4(h[0] | (h[1] << 16), h[2] | (h[3] << 16), h[4] | (h[5] << 16), h[6] | (h[7] << 16));
        }
    }
    float sq = 0.f;  // this thread's 32 values, in a fixed order
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        const int v = threadIdx.x + t * kPrepThreads;
        const int a = v >> 3, b0 = (v & 7) * 8;
        const uint32_t w[4] = {raw[t].x, raw[t].y, raw[t].z, raw[t].w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float lo = __uint_as_float(w[k] << 16), hi = __uint_as_float(w[k] & 0xFFFF0000u);
            sq = fmaf(lo, lo, sq);
            sq = fmaf(hi, hi, sq);
        }
        if (!tr) {
            *reinterpret_cast<uint4*>(&T[a][tx(a, b0)]) = raw[t];
        } else {
#pragma unroll
            for (int k = 0; k < 8; ++k)
                T[b0 + k][tx(b0 + k, a)] = static_cast<uint16_t>(k & 1 ? w[k >> 1] >> 16 : w[k >> 1] & 0xFFFFu);
        }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = sq;
    __syncthreads();
    if (threadIdx.x == 0) {
        float tot = 0.f;
#pragma unroll
        for (int k = 0; k < kPrepThreads / 32; ++k) tot += red[k];
        partials[static_cast<int64_t>(unit) * gridDim.x * gridDim.y + blockIdx.y * gridDim.x + blockIdx.x] = tot;
    }
    uint16_t* xo = X + static_cast<int64_t>(unit) * gridDim.y * 64 * np;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        const int v = threadIdx.x + t * kPrepThreads;
        const int ii = v >> 3, jj = (v & 7) * 8;
        *reinterpret_cast<uint4*>(xo + static_cast<int64_t>(i0 + ii) * np + j0 + jj) =
            *reinterpret_cast<const uint4*>(&T[ii][tx(ii, jj)]);
    }
}

__device__ __forceinline__ uint32_t bf16_rne_bits(float x) { return __bfloat16_as_ushort(__float2bfloat16_rn(x)); }

// ---------------------------------------------------------------------------
// f0 folded into the prepare pass (u as scratch): each 8-element chunk of u is
// computed from the main gradient and the momentum where they live in the
// rank segments (m <- mu*m + g, multiply then add, each rounded; u =
// bf16_RNE(m), or bf16_RNE(g + mu*m) with Nesterov -- f0's arithmetic), m is
// written back, and u goes straight into X0 with the same tile mapping,
// transposition and per-tile sums of squares as ns_prepare_kernel, so the
// norm and X0 are bit-identical to preparing from a stored u.  u itself is
// never written.  A chunk's elements lie in one fragment when u's row length
// is a multiple of 8 (fragments start on multiples of 32 unit elements);
// otherwise every element looks its fragment up.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kPrepThreads) f0_prepare_kernel(const NsUnit* __restrict__ units,
                                                                   const NsFrag* __restrict__ frags,
                                                                   float* __restrict__ m_root,
                                                                   const float* __restrict__ g_root, float mu,
                                                                   int nesterov, float* __restrict__ partials,
                                                                   uint16_t* __restrict__ X, int m, int n, int np) {
    __shared__ __align__(16) uint16_t T[64][64];
    __shared__ float red[kPrepThreads / 32];
    auto tx = [](int r, int c) { return ((((c >> 3) ^ (r >> 3)) & 7) << 3) | (c & 7); };
    const int unit = blockIdx.z;
    const NsUnit nu = units[unit];
    const bool tr = nu.flags & kNsTransposed;
    const int i0 = blockIdx.y * 64, j0 = blockIdx.x * 64;
    const int ld = tr ? m : n;
    const bool vec_ok = (ld & 7) == 0;
    const int rlim = tr ? n : m, clim = tr ? m : n;
    const NsFrag* fr = frags + nu.frag0;
    const int nf = nu.nfrag;
    const int64_t base1 = nf == 1 ? fr[0].root_off - fr[0].unit_off : -1;
    auto root_of = [&](int64_t e) -> int64_t {
        if (base1 >= 0) return base1 + e;
        int f = 0;
        while (f + 1 < nf && fr[f + 1].unit_off <= e) ++f;
        return fr[f].root_off + (e - fr[f].unit_off);
    };
    auto f0_of = [&](float g, float& mv) {  // returns u (as float) and updates m
        mv = __fadd_rn(__fmul_rn(mu, mv), g);
        return nesterov ? __fadd_rn(g, __fmul_rn(mu, mv)) : mv;
    };
    // loads of all four chunks first
    float4 gv[4][2], mv[4][2];
    int64_t ro[4];
    bool full[4];
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        const int v = threadIdx.x + t * kPrepThreads;
        const int a = v >> 3, b0 = (v & 7) * 8;
        const int ur = (tr ? j0 : i0) + a, uc = (tr ? i0 : j0) + b0;
        full[t] = ur < rlim && vec_ok && uc + 8 <= clim;
        ro[t] = 0;
        if (full[t]) {
            ro[t] = root_of(static_cast<int64_t>(ur) * ld + uc);
            const float4* gp = reinterpret_cast<const float4*>(g_root + ro[t]);
            const float4* mp = reinterpret_cast<const float4*>(m_root + ro[t]);
            gv[t][0] = __ldcs(gp);
            gv[t][1] = __ldcs(gp + 1);
            mv[t][0] = __ldcs(mp);
            mv[t][1] = __ldcs(mp + 1);
        }
    }
    uint4 raw[4];  // 8 bf16 of u per chunk, zero outside the unit
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        const int v = threadIdx.x + t * kPrepThreads;
        const int a = v >> 3, b0 = (v & 7) * 8;
        const int ur = (tr ? j0 : i0) + a, uc = (tr ? i0 : j0) + b0;
        if (full[t]) {
            const float g8[8] = {gv[t][0].x, gv[t][0].y, gv[t][0].z, gv[t][0].w,
                                 gv[t][1].x, gv[t][1].y, gv[t][1].z, gv[t][1].w};
            float m8[8] = {mv[t][0].x, mv[t][0].y, mv[t][0].z, mv[t][0].w, mv[t][1].x, mv[t][1].y, mv[t][1].z, mv[t][1].w};
            float u8[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) u8[k] = f0_of(g8[k], m8[k]);
            float4* mp = reinterpret_cast<float4*>(m_root + ro[t]);
            __stcs(mp, make_float4(m8[0], m8[1], m8[2], m8[3]));
            __stcs(mp + 1, make_float4(m8[4], m8[5], m8[6], m8[7]));
            raw[t] = make_uint4(bf16_rne_bits(u8[0]) | (bf16_rne_bits(u8[1]) << 16), bf16_rne_bits(u8[2]) | (bf16_rne_bits(u8[3]) << 16),
                                bf16_rne_bits(u8[4]) | (bf16_rne_bits(u8[5]) << 16), bf16_rne_bits(u8[6]) | (bf16_rne_bits(u8[7]) << 16));
        } else {
            uint32_t h[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                h[k] = 0u;
                if (ur < rlim && uc + k < clim) {
                    const int64_t r = root_of(static_cast<int64_t>(ur) * ld + uc + k);
                    float mk = m_root[r];
                    const float uk = f0_of(g_root[r], mk);
                    m_root[r] = mk;
                    h[k] = bf16_rne_bits(uk);
                }
            }
            raw[t] = make_uint4(h[0] | (h[1] << 16), h[2] | (h[3] << 16), h[4] | (h[5] << 16), h[6] | (h[7] << 16));
        }
    }
    float sq = 0.f;  // this thread's 32 values, in a fixed order (that of ns_prepare_kernel)
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        const int v = threadIdx.x + t * kPrepThreads;
        const int a = v >> 3, b0 = (v & 7) * 8;
        const uint32_t w[4] = {raw[t].x, raw[t].y, raw[t].z, raw[t].w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float lo = __uint_as_float(w[k] << 16), hi = __uint_as_float(w[k] & 0xFFFF0000u);
            sq = fmaf(lo, lo, sq);
            sq = fmaf(hi, hi, sq);
        }
        if (!tr) {
            *reinterpret_cast<uint4*>(&T[a][tx(a, b0)]) = raw[t];
        } else {
#pragma unroll
            for (int k = 0; k < 8; ++k)
                T[b0 + k][tx(b0 + k, a)] = static_cast<uint16_t>(k & 1 ? w[k >> 1] >> 16 : w[k >> 1] & 0xFFFFu);
        }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = sq;
    __syncthreads();
    if (threadIdx.x == 0) {
        float tot = 0.f;
#pragma unroll
        for (int k = 0; k < kPrepThreads / 32; ++k) tot += red[k];
        partials[static_cast<int64_t>(unit) * gridDim.x * gridDim.y + blockIdx.y * gridDim.x + blockIdx.x] = tot;
    }
    uint16_t* xo = X + static_cast<int64_t>(unit) * gridDim.y * 64 * np;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        const int v = threadIdx.x + t * kPrepThreads;
        const int ii = v >> 3, jj = (v & 7) * 8;
        *reinterpret_cast<uint4*>(xo + static_cast<int64_t>(i0 + ii) * np + j0 + jj) =
            *reinterpret_cast<const uint4*>(&T[ii][tx(ii, jj)]);
    }
}

// ---------------------------------------------------------------------------
// PTX wrappers: mbarrier, TMA, tcgen05
// ---------------------------------------------------------------------------
constexpr int BM = 128;
constexpr int BK = 64;
constexpr int kEpiWarps = 8;  // two per TMEM lane quadrant, each drains half of a tile's columns
constexpr int kGemmThreads = 64 + 32 * kEpiWarps;
constexpr unsigned long long kWaitNs = 2000000000ull;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ unsigned long long globaltimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait.  Gives up when another role of the CTA has given up (bail)
// or after kWaitNs; the first give-up records HM_ERR_TIMEOUT.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, int32_t* err, volatile int* bail,
                                          bool honour_bail = true) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer();
    while (true) {
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (honour_bail && *bail) return false;
        if (globaltimer() - t0 > kWaitNs) {
            *bail = 1;
            if (err) atomicCAS(err, 0, kDevErrTimeout);
            return false;
        }
    }
}
// Pacing of the CTA pairs.  Tiles are dealt round-robin, so in wave k every
// pair works on its k-th tile and tiles that share an operand panel run at
// the same time; left alone, pairs drift apart over many waves and those
// panels come from DRAM again.  Each pair's producer counts the tiles whose
// loads it has issued in pace[0] and, before its k-th tile, waits until
// every pair has issued its (k-1)-th.  The wait only shapes timing: it gives
// up after kPaceWaitNs and carries on, so it can neither hang nor change a
// result.  The last pair to finish zeroes both counters for the next launch.
constexpr unsigned long long kPaceWaitNs = 200000;  // 200 us

__device__ __forceinline__ void pace_wait(const int32_t* issued, int target) {
    if (*reinterpret_cast<const volatile int32_t*>(issued) >= target) return;
    const unsigned long long t0 = globaltimer();
    while (*reinterpret_cast<const volatile int32_t*>(issued) < target)
        if (globaltimer() - t0 > kPaceWaitNs) return;
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int c0, int c1,
                                            int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void umma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
// After tmem_ld_wait: makes every later use of r depend on a point after the
// wait, so the compiler cannot read registers a tcgen05.ld is still filling.
__device__ __forceinline__ void tmem_ld_pin(uint32_t (&r)[32]) {
    asm volatile(""
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                   "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                   "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]),
                   "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]),
                   "+r"(r[29]), "+r"(r[30]), "+r"(r[31]));
}

// Shared-memory matrix descriptor of a K-major operand tile written by TMA
// with the 128-byte swizzle: rows of 64 bf16 (128 B), 8-row atoms of 1024 B
// (stride-dimension byte offset 1024), descriptor version 1, swizzle mode
// "128B".  Advancing K by 16 elements adds 32 bytes to the start address.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
    return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>(1) << 16) |
           (static_cast<uint64_t>(1024 >> 4) << 32) | (static_cast<uint64_t>(1) << 46) |
           (static_cast<uint64_t>(2) << 61);
}

// The same for an MN-major operand (N contiguous) loaded as BN/64 TMA boxes of
// 64 N x 64 K, each box 64 rows (one per K) of 128 B: 8-K-row atoms of 1024 B
// (stride-dimension byte offset 1024), consecutive 64-element N chunks 8 KiB
// apart (leading-dimension byte offset 8192).  Advancing K by 16 rows adds
// 2048 bytes to the start address.
__device__ __forceinline__ uint64_t desc_mn_sw128(uint32_t saddr) {
    return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>(8192 >> 4) << 16) |
           (static_cast<uint64_t>(1024 >> 4) << 32) | (static_cast<uint64_t>(1) << 46) |
           (static_cast<uint64_t>(2) << 61);
}

template <int BN, bool B_MN>
struct GemmCfg {
    static constexpr int STAGES = BN == 256 ? 4 : 6;
    static constexpr int A_BYTES = BM * BK * 2;
    static constexpr int B_BYTES = BN * BK * 2;
    static constexpr int TMEM_COLS = 2 * BN;
    static constexpr int EPI_BYTES = kEpiWarps * 32 * 33 * 4;  // per epilogue warp: a 32 x 32 fp32 transpose tile
    static constexpr int SMEM = STAGES * (A_BYTES + B_BYTES) + EPI_BYTES + 1024 + 256;
    // kind::f16 instruction descriptor: D fp32, A and B bf16, A K-major, B
    // K-major or (bit 16) MN-major, N >> 3 at bit 17, M >> 4 at bit 24.
    static constexpr uint32_t IDESC = (1u << 4) | (1u << 7) | (1u << 10) | (B_MN ? (1u << 16) : 0u) |
                                      (static_cast<uint32_t>(BN >> 3) << 17) |
                                      (static_cast<uint32_t>(BM >> 4) << 24);
    // descriptor start-address step (16-byte units) per K = 16 MMA
    static constexpr uint64_t B_KSTEP = B_MN ? (2048 >> 4) : (32 >> 4);
};

__device__ __forceinline__ void decode_tile(int t, const GemmParams& p, int& u, int& tm, int& tn) {
    if (p.tile_tab) {
        u = t / p.tab_len;
        const int32_t e = __ldg(p.tile_tab + (t - u * p.tab_len));
        tm = e >> 16;
        tn = e & 0xFFFF;
        return;
    }
    const int per = p.tiles_m * p.tiles_n;
    u = t / per;
    const int r = t - u * per;
    const int band = p.group_m > 0 ? p.group_m : 8;
    const int group = band * p.tiles_n;
    const int g = r / group;
    const int first = g * band;
    const int gm = min(p.tiles_m - first, band);
    const int rr = r - g * group;
    tm = first + rr % gm;
    tn = rr / gm;
}

__device__ __forceinline__ void unpack_bf16x8(const uint4& x, float* f) {
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        f[2 * k] = __uint_as_float(w[k] << 16);
        f[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
    }
}
__device__ __forceinline__ uint32_t bf16_bits(float x) { return __bfloat16_as_ushort(__float2bfloat16_rn(x)); }
// Two floats rounded to bf16 (RNE) in one conversion; lo in the low half.
__device__ __forceinline__ uint32_t bf16x2_bits(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
}

// Epilogues that add aX read the addend with 4 lanes per row (see below).
__device__ __forceinline__ bool addend_coalesced(const GemmParams& p) {
    return ((p.epi == kEpiUpdate || p.epi == kEpiFinal) && !p.sym) || (p.epi == kEpiPoly && p.sym);
}

// With a short K (B X of the 128-row head class: two k-blocks) the epilogue,
// not the MMA, sets the pace, so the first addend chunk of a tile is loaded
// before its accumulator is ready.  With a long K the addend is left until
// the accumulator is ready: by then the tile's TMA loads have brought those
// rows of X into the L2, and an early read would fetch them from DRAM.
constexpr int kEarlyAddendKb = 8;

// Loads one 32 x 32 chunk of the addend X (rows i0.., columns j0..) in the
// coalesced pattern: lane l holds row i0 + l/4 + 8s, columns j0 + 8(l%4)..+7.
__device__ __forceinline__ void load_addend_chunk(const GemmParams& p, int u, int i0, int j0, uint4 (&a)[4]) {
    const int lane = threadIdx.x & 31;
    if (j0 >= p.N) return;
    const uint16_t* ab = p.add + u * p.add_us + j0 + (lane & 3) * 8;
#pragma unroll
    for (int s = 0; s < 4; ++s)
        a[s] = __ldg(reinterpret_cast<const uint4*>(ab + static_cast<int64_t>(i0 + (lane >> 2) + 8 * s) * p.ld_add));
}

// The fragment of a kNsEpiUpdate unit that holds unit element e (a block start).
__device__ __forceinline__ int64_t unit_root_offset(const GemmParams& p, const NsUnit& nu, int64_t e) {
    int f = nu.frag0;
    while (f + 1 < nu.frag0 + nu.nfrag && p.frags[f + 1].unit_off <= e) ++f;
    return p.frags[f].root_off + (e - p.frags[f].unit_off);
}

// A warp's 32 x 32 fp32 staging tile keeps 16-byte chunk c4 of row r at
// chunk c4 ^ swz(r), swz(r) = (r % 8) ^ 2 (r / 8): the row-wise writes (lane r
// writes row r), the 4-lanes-per-row reads (lanes 4k..4k+3 read row k + 8s)
// and the column reads of the mirror and transposed paths (lane reads column
// l/4 + 8s of rows 8(l%4) + e) all hit 32 distinct banks.
__device__ __forceinline__ int swz(int r) { return (r & 7) ^ ((r >> 2) & 6); }
__device__ __forceinline__ float4* stage4(float* stage, int r, int c4) {
    return reinterpret_cast<float4*>(stage + r * 32 + ((c4 ^ swz(r)) << 2));
}
__device__ __forceinline__ float4 stage4_ld(const float* stage, int r, int c4) {
    return *reinterpret_cast<const float4*>(stage + r * 32 + ((c4 ^ swz(r)) << 2));
}
// element (r, c) of the staging tile
__device__ __forceinline__ float stage_at(const float* stage, int r, int c) {
    return stage[r * 32 + ((((c >> 2) ^ swz(r)) << 2) | (c & 3))];
}
// column c of rows r0 .. r0+7 (r0 a multiple of 8, so swz(r0 + e) = e ^ r0 / 4)
__device__ __forceinline__ void stage_col8(const float* stage, int r0, int c, float (&y)[8]) {
    const int k0 = (c >> 2) ^ (r0 >> 2);
    const float* base = stage + r0 * 32 + (c & 3);
#pragma unroll
    for (int e = 0; e < 8; ++e) y[e] = base[e * 32 + ((k0 ^ e) << 2)];
}

// staging += beta * addend (the aX term of the last product), in the layout
// of load_addend_chunk: lane l holds row l/4 + 8s, columns 8(l%4)..+7; the sum
// is scaled by sc when the product carries the first iteration's unit scale.
__device__ __forceinline__ void stage_add_addend(const GemmParams& p, float* stage, const uint4 (&a)[4], float sc) {
    const int lane = threadIdx.x & 31;
    const int cq = (lane & 3) * 8;
#pragma unroll
    for (int s = 0; s < 4; ++s) {
        const int rr = (lane >> 2) + 8 * s;
        float a8[8];
        unpack_bf16x8(a[s], a8);
        float4* p0 = stage4(stage, rr, cq >> 2);
        float4* p1 = stage4(stage, rr, (cq >> 2) + 1);
        const float4 y0 = *p0, y1 = *p1;
        float4 z0 = make_float4(fmaf(p.beta, a8[0], y0.x), fmaf(p.beta, a8[1], y0.y), fmaf(p.beta, a8[2], y0.z),
                                fmaf(p.beta, a8[3], y0.w));
        float4 z1 = make_float4(fmaf(p.beta, a8[4], y1.x), fmaf(p.beta, a8[5], y1.y), fmaf(p.beta, a8[6], y1.z),
                                fmaf(p.beta, a8[7], y1.w));
        if (p.unit_scale) {
            z0 = make_float4(z0.x * sc, z0.y * sc, z0.z * sc, z0.w * sc);
            z1 = make_float4(z1.x * sc, z1.y * sc, z1.z * sc, z1.w * sc);
        }
        *p0 = z0;
        *p1 = z1;
    }
}

// Root offsets of the four 1 x 32 blocks of w this lane works on in the chunk
// (rows i0.., columns j0.. of X): lane l takes block l/4 + 8s, elements
// 8(l%4)..+7; -1 for a row of w beyond the unit.  False when the chunk lies in
// X's zero padding (warp-uniform).
__device__ __forceinline__ bool chunk_w_blocks(const GemmParams& p, const NsUnit& nu, int64_t base1, int i0, int j0,
                                               int64_t (&dst)[4]) {
    const int lane = threadIdx.x & 31;
    const bool tr = nu.flags & kNsTransposed;
    const int kw = tr ? p.m_real : p.n_real;      // length of a row of w (the MX K)
    const int rows_w = tr ? p.n_real : p.m_real;  // rows of w
    const int rw0 = tr ? j0 : i0;                  // w row of the chunk's block 0
    const int cw0 = tr ? i0 : j0;                  // w column of every block's first element
    if (cw0 >= kw) return false;                   // padding of X
#pragma unroll
    for (int s = 0; s < 4; ++s) {
        const int rw = rw0 + (lane >> 2) + 8 * s;
        dst[s] = -1;
        if (rw >= rows_w) continue;
        // the unit's fragment that holds this block (32-aligned: the whole block)
        const int64_t e = static_cast<int64_t>(rw) * kw + cw0;
        dst[s] = base1 >= 0 ? base1 + e : unit_root_offset(p, nu, e);
    }
    return true;
}

// v of this lane's part of block s of the chunk, from the warp's staging tile
__device__ __forceinline__ void staged_block(const float* stage, bool tr, int s, float (&y)[8]) {
    const int lane = threadIdx.x & 31;
    const int cq = (lane & 3) * 8;
    const int kk = (lane >> 2) + 8 * s;
    if (tr) {
        stage_col8(stage, cq, kk, y);  // column kk of the chunk, rows cq..cq+7
    } else {
        const float4 a = stage4_ld(stage, kk, cq >> 2);
        const float4 b = stage4_ld(stage, kk, (cq >> 2) + 1);
        y[0] = a.x; y[1] = a.y; y[2] = a.z; y[3] = a.w;
        y[4] = b.x; y[5] = b.y; y[6] = b.z; y[7] = b.w;
    }
}

// Last product with the update folded in (units flagged kNsEpiUpdate): the
// chunk's 32 x 32 values of v = aX + BX (fp32, in the warp's swizzled staging
// tile) never reach memory.  Each 1 x 32 MX block of the unit's w that the
// chunk covers -- a row of the chunk, or a column when the unit is stored
// transposed (X = u^T) -- is read from the root, updated as f2 does it
// (w*decay - step*v, or w - step*v, each product and the difference rounded
// once) and quantized as G does it, so w, q and s come out bit-identical to
// the pass through v.  Four lanes own one block, 8 elements each (lane l:
// block l/4 + 8s, elements 8(l%4)..+7); the loads of all four blocks go first.
// (Issuing them before the aX addend is folded in, or a tile ahead as L2
// prefetches, measured no faster.)
//
// base1: root offset minus unit offset of a unit with one fragment (a local
// unit), read once per tile; -1 = look the fragment up per block.
__device__ __forceinline__ void final_update_chunk(const GemmParams& p, const NsUnit& nu, int64_t base1,
                                                   const float* stage, int i0, int j0) {
    const int lane = threadIdx.x & 31;
    const bool tr = nu.flags & kNsTransposed;
    const int kw = tr ? p.m_real : p.n_real;      // length of a row of w (the MX K)
    const int rows_w = tr ? p.n_real : p.m_real;  // rows of w
    const int rw0 = tr ? j0 : i0;                  // w row of the chunk's block 0
    const int cw0 = tr ? i0 : j0;                  // w column of every block's first element
    if (cw0 >= kw) return;                         // padding of X (warp-uniform)
    const int cq = (lane & 3) * 8;
    int64_t dst[4];
    float4 w0[4], w1[4];
#pragma unroll
    for (int s = 0; s < 4; ++s) {
        const int rw = rw0 + (lane >> 2) + 8 * s;
        w0[s] = w1[s] = make_float4(0.f, 0.f, 0.f, 0.f);
        dst[s] = -1;
        if (rw >= rows_w) continue;
        // the unit's fragment that holds this block (32-aligned: the whole block)
        const int64_t e = static_cast<int64_t>(rw) * kw + cw0;
        dst[s] = base1 >= 0 ? base1 + e : unit_root_offset(p, nu, e);
        const float4* wp = reinterpret_cast<const float4*>(p.w + dst[s] + cq);
        w0[s] = __ldcs(wp);
        w1[s] = __ldcs(wp + 1);
    }
#pragma unroll
    for (int s = 0; s < 4; ++s) {
        const int kk = (lane >> 2) + 8 * s;
        float y[8];
        if (tr) {
            stage_col8(stage, cq, kk, y);  // column kk of the chunk, rows cq..cq+7
        } else {
            const float4 a = stage4_ld(stage, kk, cq >> 2);
            const float4 b = stage4_ld(stage, kk, (cq >> 2) + 1);
            y[0] = a.x; y[1] = a.y; y[2] = a.z; y[3] = a.w;
            y[4] = b.x; y[5] = b.y; y[6] = b.z; y[7] = b.w;
        }
        const float wv[8] = {w0[s].x, w0[s].y, w0[s].z, w0[s].w, w1[s].x, w1[s].y, w1[s].z, w1[s].w};
        float x[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const float a = p.has_decay ? __fmul_rn(wv[e], p.decay) : wv[e];
            x[e] = __fsub_rn(a, __fmul_rn(nu.step, y[e]));
        }
        float amax = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(x[e]));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
        if (dst[s] < 0) continue;  // a row of w beyond the unit (same for the block's 4 lanes)
        float4* wp = reinterpret_cast<float4*>(p.w + dst[s] + cq);
        __stcs(wp, make_float4(x[0], x[1], x[2], x[3]));
        __stcs(wp + 1, make_float4(x[4], x[5], x[6], x[7]));
        const int ex = mx_scale_exponent(amax);
        const float sc = mx_inv_scale(ex);
        const uint32_t c01 = cvt_e4m3x2(x[0] * sc, x[1] * sc);
        const uint32_t c23 = cvt_e4m3x2(x[2] * sc, x[3] * sc);
        const uint32_t c45 = cvt_e4m3x2(x[4] * sc, x[5] * sc);
        const uint32_t c67 = cvt_e4m3x2(x[6] * sc, x[7] * sc);
        __stcs(reinterpret_cast<uint2*>(p.q + dst[s] + cq), make_uint2(c01 | (c23 << 16), c45 | (c67 << 16)));
        if ((lane & 3) == 0) p.s[dst[s] >> 5] = static_cast<uint8_t>(ex + 127);
    }
}

// The last product's 32 x 32 chunk (rows i0.., columns j0.. of X; this lane's
// row is i), parked in the warp's staging tile as fp32 values of aX + BX:
// f2 and G of the unit straight from the staging (fuse), or v written to the
// unit's own v location.
__device__ __forceinline__ void store_final_chunk(const GemmParams& p, const NsUnit& nu, bool fuse, int64_t base1,
                                                  const float* stage, int i, int i0, int j0) {
    if (fuse) {
        final_update_chunk(p, nu, base1, stage, i0, j0);
        return;
    }
    const int lane = threadIdx.x & 31;
    float* dst = ((nu.flags & kNsVStaged) ? p.v_stage : p.v_root) + nu.v_off;
    if (nu.flags & kNsTransposed) {
        // v is X^T: for each k the 32 lanes write 32 consecutive floats
        // of v's row j0 + k
        if (i < p.m_real) {
#pragma unroll
            for (int c4 = 0; c4 < 8; ++c4) {
                const float4 y = stage4_ld(stage, lane, c4);
                const float yk[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (j0 + 4 * c4 + e < p.n_real)
                        __stcs(dst + static_cast<int64_t>(j0 + 4 * c4 + e) * p.m_real + i, yk[e]);
            }
        }
    } else if (j0 + 32 <= p.n_real && (p.n_real & 3) == 0 && (reinterpret_cast<uintptr_t>(dst) & 15u) == 0) {
        // row-major v: 8 lanes per row, 16 bytes each, so every store covers
        // 4 rows x 128 contiguous bytes; streaming stores, since v is read
        // back only by f2 after the whole Newton-Schulz stage
        const int c4 = lane & 7;
#pragma unroll 1
        for (int s2 = 0; s2 < 8; ++s2) {
            const int r2 = s2 * 4 + (lane >> 3);
            if (i0 + r2 < p.m_real)
                __stcs(reinterpret_cast<float4*>(dst + static_cast<int64_t>(i0 + r2) * p.n_real + j0 + 4 * c4),
                       stage4_ld(stage, r2, c4));
        }
    } else if (j0 + lane < p.n_real) {
        // ragged or unaligned rows: one 4-byte store per lane, 128 bytes of one row per store
#pragma unroll 4
        for (int r2 = 0; r2 < 32; ++r2)
            if (i0 + r2 < p.m_real)
                dst[static_cast<int64_t>(i0 + r2) * p.n_real + j0 + lane] = stage_at(stage, r2, lane);
    }
}

// i_base: first output row of this CTA's 128-row slab of the tile.  `next`
// holds the addend of the warp's first chunk when addend_coalesced(p): the
// caller loads it before waiting for the accumulator, and each chunk loads
// the next one's before it works on its own.
template <int BN>
__device__ __forceinline__ void epilogue_tile(const GemmParams& p, int u, int i_base, int tn, int row, uint32_t taddr,
                                              float* stage, int half, uint4 (&next)[4]) {
    const int i = i_base + row;
    const int c_end = (half + 1) * (BN / 64);
    // first iteration: the unit's scale s (Gram outputs take s^2)
    const float usc = p.unit_scale ? p.unit_scale[u] : 1.f;
    const float alpha_t = p.unit_scale ? p.alpha * (usc * usc) : p.alpha;
    // last product: the unit's destination once per tile
    NsUnit nu{};
    bool fuse = false;
    int64_t base1 = -1;
    if (p.epi == kEpiFinal) {
        nu = p.ns_units[u];
        fuse = p.fuse_update && (nu.flags & kNsEpiUpdate);
        if (fuse && nu.nfrag == 1) base1 = p.frags[nu.frag0].root_off - p.frags[nu.frag0].unit_off;
    }
    // the next chunk's TMEM load is in flight while the current chunk is processed
    uint32_t rn[32];
    __syncwarp();
    tmem_ld32(taddr + half * (BN / 64) * 32, rn);
#pragma unroll 1
    for (int c = half * (BN / 64); c < c_end; ++c) {
        const int j0 = tn * BN + c * 32;
        uint4 a[4] = {next[0], next[1], next[2], next[3]};
        if (addend_coalesced(p) && c + 1 < c_end) load_addend_chunk(p, u, i - (threadIdx.x & 31), j0 + 32, next);
        tmem_ld_wait();
        tmem_ld_pin(rn);
        uint32_t r[32];
#pragma unroll
        for (int k = 0; k < 32; ++k) r[k] = rn[k];
        __syncwarp();
        if (c + 1 < c_end) tmem_ld32(taddr + (c + 1) * 32, rn);
        if (j0 >= p.N) continue;  // warp-uniform; N is a multiple of 32
        const int i0 = i - (threadIdx.x & 31);  // first row of this warp
        if (p.sym && j0 + 32 <= i0) continue;   // symmetric output: chunk below the diagonal
        if ((p.epi == kEpiUpdate || p.epi == kEpiFinal) && !p.sym) {
            // aX + BX through the warp's staging: the lane that holds row i parks
            // its 32 sums, then every load of the addend (and every store of X')
            // covers 8 rows x 64 contiguous bytes, 4 lanes per row, instead of
            // 32 rows x 16 bytes; the tile's swizzle (swz above) keeps the row-wise
            // writes and the 4-lanes-per-row reads conflict-free 16-byte accesses.
            // (These two epilogues have no alpha: acc is B X as it stands.)
            const int lane = threadIdx.x & 31;
            auto st4 = [&](int r, int c4) { return stage4(stage, r, c4); };
#pragma unroll
            for (int c4 = 0; c4 < 8; ++c4)
                *st4(lane, c4) = make_float4(__uint_as_float(r[4 * c4]), __uint_as_float(r[4 * c4 + 1]),
                                             __uint_as_float(r[4 * c4 + 2]), __uint_as_float(r[4 * c4 + 3]));
            __syncwarp();
            const int cq = (lane & 3) * 8;
            if (p.epi == kEpiUpdate) {
                uint16_t* ob = p.out + u * p.out_us + j0 + cq;
#pragma unroll
                for (int s = 0; s < 4; ++s) {
                    const int rr = (lane >> 2) + 8 * s;
                    float a8[8], o[8];
                    unpack_bf16x8(a[s], a8);
                    const float4 y0 = *st4(rr, cq >> 2), y1 = *st4(rr, (cq >> 2) + 1);
                    const float y[8] = {y0.x, y0.y, y0.z, y0.w, y1.x, y1.y, y1.z, y1.w};
#pragma unroll
                    for (int t = 0; t < 8; ++t) o[t] = fmaf(p.beta, a8[t], y[t]);
                    if (p.unit_scale) {
#pragma unroll
                        for (int t = 0; t < 8; ++t) o[t] *= usc;
                    }
                    *reinterpret_cast<uint4*>(ob + static_cast<int64_t>(i0 + rr) * p.ld_out) = make_uint4(
                        bf16x2_bits(o[0], o[1]), bf16x2_bits(o[2], o[3]),
                        bf16x2_bits(o[4], o[5]), bf16x2_bits(o[6], o[7]));
                }
                continue;
            }
            // last iteration: v = fp32(aX + BX) into the unit's own v location,
            // or f2 and G of the unit straight from the staging
            stage_add_addend(p, stage, a, usc);
            __syncwarp();
            store_final_chunk(p, nu, fuse, base1, stage, i, i0, j0);
            __syncwarp();
            continue;
        }
        if (p.sym) {
            // symmetric output (A = X X^T, B = bA + cAA): this warp owns rows
            // i0..i0+31 and writes only elements with j >= i, each to (i, j) and
            // to (j, i), through the same swizzled staging tile: the chunk and its
            // transpose both leave as 16-byte stores of 8 rows x 16 bytes
            const int lane = threadIdx.x & 31;
            auto st4 = [&](int r, int c4) { return stage4(stage, r, c4); };
#pragma unroll
            for (int c4 = 0; c4 < 8; ++c4)
                *st4(lane, c4) = make_float4(__uint_as_float(r[4 * c4]) * alpha_t, __uint_as_float(r[4 * c4 + 1]) * alpha_t,
                                             __uint_as_float(r[4 * c4 + 2]) * alpha_t,
                                             __uint_as_float(r[4 * c4 + 3]) * alpha_t);
            __syncwarp();
            const int cq = (lane & 3) * 8;
            if (p.epi == kEpiPoly) {
                // + b A, A read 4 lanes per row (prefetched like the aX addend)
#pragma unroll
                for (int s = 0; s < 4; ++s) {
                    const int rr = (lane >> 2) + 8 * s;
                    float a8[8];
                    unpack_bf16x8(a[s], a8);
                    float4* p0 = st4(rr, cq >> 2);
                    float4* p1 = st4(rr, (cq >> 2) + 1);
                    const float4 y0 = *p0, y1 = *p1;
                    *p0 = make_float4(fmaf(p.beta, a8[0], y0.x), fmaf(p.beta, a8[1], y0.y), fmaf(p.beta, a8[2], y0.z),
                                      fmaf(p.beta, a8[3], y0.w));
                    *p1 = make_float4(fmaf(p.beta, a8[4], y1.x), fmaf(p.beta, a8[5], y1.y), fmaf(p.beta, a8[6], y1.z),
                                      fmaf(p.beta, a8[7], y1.w));
                }
                __syncwarp();
            }
            uint16_t* ob = p.out + u * p.out_us;
            if (j0 == i0) {
                // the diagonal 32 x 32 block, element by element
#pragma unroll
                for (int c4 = 0; c4 < 8; ++c4) {
                    const float4 y = *st4(lane, c4);
                    const float yk[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int k = 4 * c4 + e;
                        if (k >= lane) {
                            const uint16_t bv = static_cast<uint16_t>(bf16_bits(yk[e]));
                            ob[static_cast<int64_t>(i0 + lane) * p.ld_out + j0 + k] = bv;
                            ob[static_cast<int64_t>(j0 + k) * p.ld_out + i0 + lane] = bv;
                        }
                    }
                }
            } else {
#pragma unroll
                for (int s = 0; s < 4; ++s) {
                    const int rr = (lane >> 2) + 8 * s;
                    const float4 y0 = *st4(rr, cq >> 2), y1 = *st4(rr, (cq >> 2) + 1);
                    *reinterpret_cast<uint4*>(ob + static_cast<int64_t>(i0 + rr) * p.ld_out + j0 + cq) = make_uint4(
                        bf16x2_bits(y0.x, y0.y), bf16x2_bits(y0.z, y0.w),
                        bf16x2_bits(y1.x, y1.y), bf16x2_bits(y1.z, y1.w));
                }
                // mirror: row j0 + kk of the output takes column kk of the chunk,
                // 8 of its rows per lane
#pragma unroll
                for (int s = 0; s < 4; ++s) {
                    const int kk = (lane >> 2) + 8 * s;
                    float y[8];
                    stage_col8(stage, cq, kk, y);
                    *reinterpret_cast<uint4*>(ob + static_cast<int64_t>(j0 + kk) * p.ld_out + i0 + cq) = make_uint4(
                        bf16x2_bits(y[0], y[1]), bf16x2_bits(y[2], y[3]),
                        bf16x2_bits(y[4], y[5]), bf16x2_bits(y[6], y[7]));
                }
            }
            __syncwarp();
            continue;
        }
        // full-grid outputs (the allocation-free entry point's A and B)
        float v[32];
#pragma unroll
        for (int k = 0; k < 32; ++k) v[k] = __uint_as_float(r[k]) * alpha_t;
        if (p.epi == kEpiPoly) {
            const uint4* ap = reinterpret_cast<const uint4*>(p.add + u * p.add_us + static_cast<int64_t>(i) * p.ld_add + j0);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                float a8[8];
                unpack_bf16x8(__ldg(ap + q), a8);
#pragma unroll
                for (int k = 0; k < 8; ++k) v[q * 8 + k] = fmaf(p.beta, a8[k], v[q * 8 + k]);
            }
        }
        uint4 pk[4];
#pragma unroll
        for (int q = 0; q < 4; ++q)
            pk[q] = make_uint4(bf16x2_bits(v[8 * q + 0], v[8 * q + 1]),
                               bf16x2_bits(v[8 * q + 2], v[8 * q + 3]),
                               bf16x2_bits(v[8 * q + 4], v[8 * q + 5]),
                               bf16x2_bits(v[8 * q + 6], v[8 * q + 7]));
        uint4* op = reinterpret_cast<uint4*>(p.out + u * p.out_us + static_cast<int64_t>(i) * p.ld_out + j0);
#pragma unroll
        for (int q = 0; q < 4; ++q) op[q] = pk[q];
    }
}

template <int BN, bool B_MN>
__global__ void __launch_bounds__(kGemmThreads, 1)
    ns_gemm_kernel(const __grid_constant__ CUtensorMap tma, const __grid_constant__ CUtensorMap tmb,
                   const __grid_constant__ GemmParams p) {
    using C = GemmCfg<BN, B_MN>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sa = smem;
    uint8_t* sb = sa + C::STAGES * C::A_BYTES;
    float* epi_stage = reinterpret_cast<float*>(sb + C::STAGES * C::B_BYTES);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sb + C::STAGES * C::B_BYTES + C::EPI_BYTES);
    uint64_t* full = bars;
    uint64_t* empty = bars + C::STAGES;
    uint64_t* tfull = bars + 2 * C::STAGES;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* bail = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&tfull[b]), 1);
            mbar_init(smem_u32(&tempty[b]), 32 * kEpiWarps);
        }
        mbar_init(smem_u32(drain), 1);
        *bail = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int total = p.units * (p.tile_tab ? p.tab_len : p.tiles_m * p.tiles_n);

    if (warp == 0) {
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0, armed = 0, armed_par = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                int u, tm, tn;
                decode_tile(t, p, u, tm, tn);
                for (int kb = 0; kb < p.num_kb; ++kb) {
                    if (!mbar_wait(smem_u32(&empty[s]), ph ^ 1u, p.err, bail)) { ok = false; break; }
                    const uint32_t fb = smem_u32(&full[s]);
                    mbar_arrive_expect_tx(fb, C::A_BYTES + C::B_BYTES);
                    tma_load_3d(smem_u32(sa + s * C::A_BYTES), &tma, fb, kb * BK, tm * BM, u);
                    if (B_MN) {
#pragma unroll
                        for (int c = 0; c < BN / 64; ++c)
                            tma_load_3d(smem_u32(sb + s * C::B_BYTES + c * 8192), &tmb, fb, tn * BN + c * 64, kb * BK,
                                        u);
                    } else {
                        tma_load_3d(smem_u32(sb + s * C::B_BYTES), &tmb, fb, kb * BK, tn * BN, u);
                    }
                    armed |= 1u << s;
                    armed_par = (armed_par & ~(1u << s)) | (ph << s);
                    if (++s == C::STAGES) { s = 0; ph ^= 1u; }
                }
            }
            // wait for this CTA's own copies still in flight
            for (int k = 0; k < C::STAGES; ++k)
                if (armed & (1u << k)) mbar_wait(smem_u32(&full[k]), (armed_par >> k) & 1u, p.err, bail, false);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            int s = 0, acc = 0;
            uint32_t ph = 0, aph = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                if (!mbar_wait(smem_u32(&tempty[acc]), aph ^ 1u, p.err, bail)) break;
                tc_fence_after();
                const uint32_t d = tmem + static_cast<uint32_t>(acc * BN);
                for (int kb = 0; kb < p.num_kb; ++kb) {
                    if (!mbar_wait(smem_u32(&full[s]), ph, p.err, bail)) { ok = false; break; }
                    tc_fence_after();
                    const uint64_t ad = desc_sw128(smem_u32(sa + s * C::A_BYTES));
                    const uint32_t bs = smem_u32(sb + s * C::B_BYTES);
                    const uint64_t bd = B_MN ? desc_mn_sw128(bs) : desc_sw128(bs);
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)
                        umma_bf16(d, ad + 2 * kk, bd + C::B_KSTEP * kk, C::IDESC, (kb | kk) != 0);
                    umma_commit(smem_u32(&empty[s]));
                    if (++s == C::STAGES) { s = 0; ph ^= 1u; }
                }
                if (!ok) break;
                if (!p.inject_no_ready) umma_commit(smem_u32(&tfull[acc]));
                acc ^= 1;
                if (!acc) aph ^= 1u;
            }
            // every MMA this thread issued has completed before TMEM is freed
            umma_commit(smem_u32(drain));
            mbar_wait(smem_u32(drain), 0, p.err, bail, false);
        }
    } else {
        const int q = warp & 3;           // TMEM lane quadrant of this warp
        const int half = (warp - 2) >> 2;  // which half of the tile's columns it drains
        const int row = q * 32 + lane;
        int acc = 0;
        uint32_t aph = 0;
        for (int t = blockIdx.x; t < total; t += gridDim.x) {
            int u, tm, tn;
            decode_tile(t, p, u, tm, tn);
            uint4 first[4] = {};
            const bool early = addend_coalesced(p) && p.num_kb <= kEarlyAddendKb;
            if (early) load_addend_chunk(p, u, tm * BM + q * 32, tn * BN + half * (BN / 2), first);
            bool ok = mbar_wait(smem_u32(&tfull[acc]), aph, p.err, bail);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            if (addend_coalesced(p) && !early)
                load_addend_chunk(p, u, tm * BM + q * 32, tn * BN + half * (BN / 2), first);
            epilogue_tile<BN>(p, u, tm * BM, tn, row,
                              tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * BN),
                              epi_stage + (warp - 2) * 32 * 33, half, first);
            tc_fence_before();
            mbar_arrive(smem_u32(&tempty[acc]));
            acc ^= 1;
            if (!acc) aph ^= 1u;
        }
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

// ---------------------------------------------------------------------------
// CTA-pair variant (cta_group::2): a cluster of two CTAs computes one
// 256 x 256 output tile.  Each CTA loads its own 128 rows of A and half of
// B (128 rows K-major, or 128 columns MN-major) into its shared memory; the
// even CTA of the pair issues tcgen05.mma.cta_group::2 (M = 256, N = 256,
// K = 16), which reads both CTAs' operands and writes rows 0-127 of D into
// the even CTA's TMEM and rows 128-255 into the odd CTA's.  Per SM this halves
// the B operand traffic of the 1-CTA 128 x 256 tile.  Barriers:
//   full[s]   even CTA only: one expect_tx for both CTAs' bytes; both CTAs'
//             TMA loads complete_tx on it (cta_group::2 TMA);
//   empty[s]  in both CTAs, arrived by the MMA commit multicast to the pair;
//   tfull[b]  in both CTAs, MMA commit multicast;
//   tempty[b] even CTA only, arrived by the epilogue threads of both CTAs.
// Every wait is bounded as in the 1-CTA kernel; a cluster barrier before the
// end keeps each CTA's shared memory alive while its peer may still read it.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const CUtensorMap* map, uint32_t bar_cluster, int c0,
                                                 int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void umma_bf16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                               uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void umma_commit_pair(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
        "h"(static_cast<uint16_t>(3))
        : "memory");
}

template <bool B_MN>
struct PairCfg {
    static constexpr int BNP = 256;                 // N of the pair tile
    static constexpr int STAGES = 6;
    static constexpr int A_BYTES = BM * BK * 2;     // this CTA's 128 rows of A
    static constexpr int B_BYTES = 128 * BK * 2;    // this CTA's half of B
    static constexpr int TMEM_COLS = 2 * BNP;
    static constexpr int EPI_BYTES = kEpiWarps * 32 * 33 * 4;
    static constexpr int SMEM = STAGES * (A_BYTES + B_BYTES) + EPI_BYTES + 1024 + 256;
    static constexpr uint32_t IDESC = (1u << 4) | (1u << 7) | (1u << 10) | (B_MN ? (1u << 16) : 0u) |
                                      (static_cast<uint32_t>(BNP >> 3) << 17) |
                                      (static_cast<uint32_t>(256 >> 4) << 24);
    static constexpr uint64_t B_KSTEP = B_MN ? (2048 >> 4) : (32 >> 4);
};

template <bool B_MN>
__global__ void __launch_bounds__(kGemmThreads, 1)
    ns_gemm_pair_kernel(const __grid_constant__ CUtensorMap tma, const __grid_constant__ CUtensorMap tmb,
                        const __grid_constant__ GemmParams p) {
    using C = PairCfg<B_MN>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sa = smem;
    uint8_t* sb = sa + C::STAGES * C::A_BYTES;
    float* epi_stage = reinterpret_cast<float*>(sb + C::STAGES * C::B_BYTES);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sb + C::STAGES * C::B_BYTES + C::EPI_BYTES);
    uint64_t* full = bars;
    uint64_t* empty = bars + C::STAGES;
    uint64_t* tfull = bars + 2 * C::STAGES;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* bail = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank() & 1u;
    const bool leader = rank == 0;
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&tfull[b]), 1);
            mbar_init(smem_u32(&tempty[b]), 2 * 32 * kEpiWarps);
        }
        mbar_init(smem_u32(drain), 1);
        *bail = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_u32(tmem_slot), C::TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    cluster_sync_all();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int per_unit = p.tile_tab ? p.tab_len : p.tiles_m * p.tiles_n;
    const int total = p.units * per_unit;
    const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;

    if (warp == 0) {
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0, armed = 0, armed_par = 0;
            bool ok = true;
            int k_local = 0;
            for (int t = pair; t < total && ok; t += npairs, ++k_local) {
                int u, tm, tn;
                decode_tile(t, p, u, tm, tn);
                if (p.pace && leader && k_local > 0) pace_wait(p.pace, k_local * npairs);
                for (int kb = 0; kb < p.num_kb; ++kb) {
                    if (!mbar_wait(smem_u32(&empty[s]), ph ^ 1u, p.err, bail)) { ok = false; break; }
                    armed |= 1u << s;
                    armed_par = (armed_par & ~(1u << s)) | (ph << s);
                    const uint32_t fb = mapa_shared(smem_u32(&full[s]), 0);
                    if (leader) mbar_arrive_expect_tx(smem_u32(&full[s]), 2 * (C::A_BYTES + C::B_BYTES));
                    tma_load_3d_pair(smem_u32(sa + s * C::A_BYTES), &tma, fb, kb * BK, tm * 256 + rank * 128, u);
                    if (B_MN) {
#pragma unroll
                        for (int c = 0; c < 2; ++c)
                            tma_load_3d_pair(smem_u32(sb + s * C::B_BYTES + c * 8192), &tmb, fb,
                                             tn * C::BNP + rank * 128 + c * 64, kb * BK, u);
                    } else {
                        tma_load_3d_pair(smem_u32(sb + s * C::B_BYTES), &tmb, fb, kb * BK, tn * C::BNP + rank * 128, u);
                    }
                    if (++s == C::STAGES) { s = 0; ph ^= 1u; }
                }
                if (p.pace && leader) atomicAdd(p.pace, 1);
            }
            if (p.pace && leader) {
                // a pair that stopped early still counts its remaining tiles,
                // so no other pair waits for them
                for (int t = pair + k_local * npairs; t < total; t += npairs) atomicAdd(p.pace, 1);
                if (atomicAdd(p.pace + 1, 1) == npairs - 1) {
                    atomicExch(p.pace, 0);
                    atomicExch(p.pace + 1, 0);
                }
            }
            // the even CTA's full barriers count both CTAs' bytes: waiting on
            // them covers every copy of the pair still in flight
            if (leader)
                for (int k = 0; k < C::STAGES; ++k)
                    if (armed & (1u << k)) mbar_wait(smem_u32(&full[k]), (armed_par >> k) & 1u, p.err, bail, false);
        }
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            int s = 0, acc = 0;
            uint32_t ph = 0, aph = 0;
            bool ok = true;
            for (int t = pair; t < total && ok; t += npairs) {
                if (!mbar_wait(smem_u32(&tempty[acc]), aph ^ 1u, p.err, bail)) break;
                tc_fence_after();
                const uint32_t d = tmem + static_cast<uint32_t>(acc * C::BNP);
                for (int kb = 0; kb < p.num_kb; ++kb) {
                    if (!mbar_wait(smem_u32(&full[s]), ph, p.err, bail)) { ok = false; break; }
                    tc_fence_after();
                    const uint64_t ad = desc_sw128(smem_u32(sa + s * C::A_BYTES));
                    const uint32_t bs = smem_u32(sb + s * C::B_BYTES);
                    const uint64_t bd = B_MN ? desc_mn_sw128(bs) : desc_sw128(bs);
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)
                        umma_bf16_pair(d, ad + 2 * kk, bd + C::B_KSTEP * kk, C::IDESC, (kb | kk) != 0);
                    umma_commit_pair(smem_u32(&empty[s]));
                    if (++s == C::STAGES) { s = 0; ph ^= 1u; }
                }
                if (!ok) break;
                if (!p.inject_no_ready) umma_commit_pair(smem_u32(&tfull[acc]));
                acc ^= 1;
                if (!acc) aph ^= 1u;
            }
            umma_commit_pair(smem_u32(drain));
            mbar_wait(smem_u32(drain), 0, p.err, bail, false);
        }
    } else {
        const int q = warp & 3;
        const int half = (warp - 2) >> 2;
        const int row = q * 32 + lane;
        const uint32_t tempty_leader0 = mapa_shared(smem_u32(&tempty[0]), 0);
        const uint32_t tempty_leader1 = mapa_shared(smem_u32(&tempty[1]), 0);
        int acc = 0;
        uint32_t aph = 0;
        for (int t = pair; t < total; t += npairs) {
            int u, tm, tn;
            decode_tile(t, p, u, tm, tn);
            const int i_base = tm * 256 + static_cast<int>(rank) * 128;
            uint4 first[4] = {};
            const bool coalesced = addend_coalesced(p) && i_base < p.M;
            const bool early = coalesced && p.num_kb <= kEarlyAddendKb;
            if (early) load_addend_chunk(p, u, i_base + q * 32, tn * C::BNP + half * (C::BNP / 2), first);
            bool ok = mbar_wait(smem_u32(&tfull[acc]), aph, p.err, bail);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            if (coalesced && !early) load_addend_chunk(p, u, i_base + q * 32, tn * C::BNP + half * (C::BNP / 2), first);
            if (i_base < p.M)  // a slab beyond the last row (M a multiple of 128) holds no output
                epilogue_tile<C::BNP>(p, u, i_base, tn, row,
                                      tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * C::BNP),
                                      epi_stage + (warp - 2) * 32 * 33, half, first);
            tc_fence_before();
            mbar_arrive_cluster(acc ? tempty_leader1 : tempty_leader0);
            acc ^= 1;
            if (!acc) aph ^= 1u;
        }
    }
    // the peer's MMAs read this CTA's shared memory and write its TMEM: keep
    // both alive until every role of both CTAs is done
    __syncwarp();
    tc_fence_before();
    cluster_sync_all();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem, C::TMEM_COLS);
    }
}

// ---------------------------------------------------------------------------
// Whole Newton-Schulz of a class whose Gram size is 128 (m <= 128: the
// per-head units) in one persistent kernel.  A CTA takes whole units (unit
// blockIdx.x, then + gridDim.x, ...) and keeps all but X on chip: A and B
// (128 x 128) live in TMEM and shared memory while X streams through a ring
// of 128-row x 64-column tiles.  Per unit:
//   Gram pass:   A = X0 X0^T, accumulated over X0's tiles;
//   iteration:   B = bA + cAA (A and B rounded to bf16 in shared memory),
//                then one pass over X's tiles: X'_j = aX_j + B X_j and --
//                except in the last iteration -- A' += X'_j X'_j^T, read
//                from the bf16 X'_j the epilogue has just written to shared
//                memory, which a TMA store also sends to the other X buffer
//                for the next pass.  The last iteration writes v, or applies
//                f2 and G, instead of storing X'.
// So X is read once per iteration and written once, where the three-launch
// form reads it in X X^T, again in B X, and writes X'.  Consecutive passes
// run in opposite tile orders, so each starts on the tiles the previous one
// touched last, which are still in the L2.  The element-wise arithmetic of
// every product is that of the three-launch epilogues; only the order in
// which A's fp32 sums are accumulated over the tiles differs.
// Roles (11 warps): warp 0 issues the TMA loads, warp 1 allocates TMEM and
// issues the MMAs, warp 2 the TMA stores of X', warps 3-10 run the
// epilogues (two per TMEM lane quadrant; for a 64-column tile each drains
// 32 columns, for A and B each 64).
// TMEM: A [0, 128), AA [128, 256), four 64-column B X accumulators [256, 512).
// Every wait is bounded, as in the GEMM kernels.
// ---------------------------------------------------------------------------
constexpr int kSmallThreads = 352;
constexpr int kSmallNB = 4;                  // B X accumulators
constexpr int kSmallTile = 128 * 64 * 2;     // a 128 x 64 bf16 tile (16 KB)
constexpr int kSmallWGroup = 1;              // w blocks updated together in the last pass (1, 2, 4 measured alike)
// CS = 1: one CTA per unit.  CS = 2: a unit's tiles split over a CTA pair (a
// cluster), for classes with fewer units than CTA pairs; each CTA accumulates
// the part of A from its tiles, and A is formed by adding the two parts over
// distributed shared memory (below).  RING: X tiles in flight; XO: X' tiles in
// shared memory (written, awaiting the A MMA and the store); LAG: how many
// tiles the A MMA of X'_j trails the B X products (LAG 2 with 4 X' tiles
// measured 2 % faster than LAG 1 with 2); RECV: the peer's half-band of A.
template <int CS> struct SmallTraits;
template <> struct SmallTraits<1> { static constexpr int RING = 4, XO = 4, LAG = 2, RECV = 0; };
template <> struct SmallTraits<2> { static constexpr int RING = 4, XO = 2, LAG = 1, RECV = 64 * 128 * 4; };
template <int CS>
struct SmallCfg {
    using T = SmallTraits<CS>;
    static_assert(T::XO >= T::LAG + 1 && T::XO >= 2, "X' buffers");
    static constexpr int RING_OFF = 0;
    static constexpr int AS_OFF = RING_OFF + T::RING * kSmallTile;     // A, bf16: two [128][64] K atoms
    static constexpr int BS_OFF = AS_OFF + 2 * kSmallTile;              // B, bf16: the same layout
    static constexpr int XO_OFF = BS_OFF + 2 * kSmallTile;              // X' tiles
    static constexpr int ST_OFF = XO_OFF + T::XO * kSmallTile;          // per epilogue warp a 32 x 32 fp32 tile
    static constexpr int RECV_OFF = ST_OFF + kEpiWarps * 32 * 32 * 4;   // CS = 2: the peer's part of this CTA's band of A
    static constexpr int BAR_OFF = RECV_OFF + T::RECV;
    static constexpr int SMEM = BAR_OFF + 512 + 1024;
    // kind::f16, D fp32, A and B bf16: M = N = 128 with both operands K-major
    // (A X X^T and A A); M = 128, N = 64 with B MN-major (B X)
    static constexpr uint32_t IDESC_G = (1u << 4) | (1u << 7) | (1u << 10) | ((128u >> 3) << 17) | ((128u >> 4) << 24);
    static constexpr uint32_t IDESC_BX =
        (1u << 4) | (1u << 7) | (1u << 10) | (1u << 16) | ((64u >> 3) << 17) | ((128u >> 4) << 24);
};

__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t src, int c0, int c1, int c2) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(src), "r"(c0), "r"(c1), "r"(c2)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void fence_async_smem_cluster() {
    asm volatile("fence.proxy.async.shared::cluster;" ::: "memory");
}
// a 16-byte store into a CTA of the cluster (addr from mapa)
__device__ __forceinline__ void st_cluster_u4(uint32_t addr, uint4 v) {
    asm volatile("st.shared::cluster.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}
// Bounded wait with cluster-scope acquire, for barriers the peer CTA arrives
// on after writing this CTA's shared memory.
__device__ __forceinline__ bool mbar_try_wait_cl(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ bool mbar_wait_cl(uint32_t bar, uint32_t parity, int32_t* err, volatile int* bail) {
    if (mbar_try_wait_cl(bar, parity)) return true;
    const unsigned long long t0 = globaltimer();
    while (true) {
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait_cl(bar, parity)) return true;
        if (*bail) return false;
        if (globaltimer() - t0 > kWaitNs) {
            *bail = 1;
            if (err) atomicCAS(err, 0, kDevErrTimeout);
            return false;
        }
    }
}
__device__ __forceinline__ void fence_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }

// 16-byte chunk c (8 bf16) of row r of a [128][64] bf16 tile written with the
// 128-byte swizzle (the layout of the TMA boxes and of the MMA operands)
__device__ __forceinline__ uint32_t tile_chunk(int r, int c) {
    return static_cast<uint32_t>(r * 128 + ((c ^ (r & 7)) << 4));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_1() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// The last product with f2 and G folded in reads w one chunk ahead: this
// lane's 8 elements of each of the chunk's four w blocks are copied
// asynchronously into the warp's 4 KB buffer (float4 (2s + half) * 32 + lane,
// so the read-back is conflict-free), then consumed a tile later.
__device__ __forceinline__ void prefetch_w_chunk(const GemmParams& p, const NsUnit& nu, int64_t base1, int i0, int j0,
                                                 uint32_t buf) {
    int64_t dst[4];
    if (!chunk_w_blocks(p, nu, base1, i0, j0, dst)) return;
    const int lane = threadIdx.x & 31;
    const int cq = (lane & 3) * 8;
#pragma unroll
    for (int s = 0; s < 4; ++s) {
        if (dst[s] < 0) continue;
        const float* src = p.w + dst[s] + cq;
        cp_async16(buf + ((2 * s) * 32 + lane) * 16, src);
        cp_async16(buf + ((2 * s + 1) * 32 + lane) * 16, src + 4);
    }
}
// G blocks at a time, interleaved: the element updates, the amax trees (max is
// exact, so the order does not matter), the shuffles and the stores of the G
// blocks are independent chains the warp can overlap.
template <int G>
__device__ __forceinline__ void update_w_group(const GemmParams& p, float step, float (&x)[G][8], const float (&wv)[G][8],
                                               const int64_t* dst, int cq) {
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const float a = p.has_decay ? __fmul_rn(wv[g][e], p.decay) : wv[g][e];
            x[g][e] = __fsub_rn(a, __fmul_rn(step, x[g][e]));
        }
    float am[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        const float m01 = fmaxf(fabsf(x[g][0]), fabsf(x[g][1])), m23 = fmaxf(fabsf(x[g][2]), fabsf(x[g][3]));
        const float m45 = fmaxf(fabsf(x[g][4]), fabsf(x[g][5])), m67 = fmaxf(fabsf(x[g][6]), fabsf(x[g][7]));
        am[g] = fmaxf(fmaxf(m01, m23), fmaxf(m45, m67));
    }
#pragma unroll
    for (int g = 0; g < G; ++g) am[g] = fmaxf(am[g], __shfl_xor_sync(0xffffffffu, am[g], 1));
#pragma unroll
    for (int g = 0; g < G; ++g) am[g] = fmaxf(am[g], __shfl_xor_sync(0xffffffffu, am[g], 2));
#pragma unroll
    for (int g = 0; g < G; ++g) {
        if (dst[g] < 0) continue;  // a row of w beyond the unit (same for the block's 4 lanes)
        float4* wp = reinterpret_cast<float4*>(p.w + dst[g] + cq);
        __stcs(wp, make_float4(x[g][0], x[g][1], x[g][2], x[g][3]));
        __stcs(wp + 1, make_float4(x[g][4], x[g][5], x[g][6], x[g][7]));
        const int ex = mx_scale_exponent(am[g]);
        const float sc = mx_inv_scale(ex);
        const uint32_t c01 = cvt_e4m3x2(x[g][0] * sc, x[g][1] * sc);
        const uint32_t c23 = cvt_e4m3x2(x[g][2] * sc, x[g][3] * sc);
        const uint32_t c45 = cvt_e4m3x2(x[g][4] * sc, x[g][5] * sc);
        const uint32_t c67 = cvt_e4m3x2(x[g][6] * sc, x[g][7] * sc);
        __stcs(reinterpret_cast<uint2*>(p.q + dst[g] + cq), make_uint2(c01 | (c23 << 16), c45 | (c67 << 16)));
        if ((threadIdx.x & 3) == 0) p.s[dst[g] >> 5] = static_cast<uint8_t>(ex + 127);
    }
}

template <int G>
__device__ __forceinline__ void final_update_chunk_buf(const GemmParams& p, const NsUnit& nu, int64_t base1,
                                                       const float* stage, int i0, int j0, const float4* buf) {
    int64_t dst[4];
    if (!chunk_w_blocks(p, nu, base1, i0, j0, dst)) return;
    const int lane = threadIdx.x & 31;
    const bool tr = nu.flags & kNsTransposed;
#pragma unroll
    for (int s0 = 0; s0 < 4; s0 += G) {
        float x[G][8], wv[G][8];  // x holds the staged v, then the new w
#pragma unroll
        for (int g = 0; g < G; ++g) {
            staged_block(stage, tr, s0 + g, x[g]);
            const float4 a = buf[(2 * (s0 + g)) * 32 + lane], b = buf[(2 * (s0 + g) + 1) * 32 + lane];
            wv[g][0] = a.x; wv[g][1] = a.y; wv[g][2] = a.z; wv[g][3] = a.w;
            wv[g][4] = b.x; wv[g][5] = b.y; wv[g][6] = b.z; wv[g][7] = b.w;
        }
        update_w_group<G>(p, nu.step, x, wv, dst + s0, (lane & 3) * 8);
    }
}

template <int CS>
__global__ void __launch_bounds__(kSmallThreads, 1)
    ns_small_kernel(const __grid_constant__ CUtensorMap tx0, const __grid_constant__ CUtensorMap tx1,
                    const __grid_constant__ SmallNsParams sp) {
    using C = SmallCfg<CS>;
    constexpr int kSmallRing = C::T::RING;
    constexpr int kSmallXo = C::T::XO;
    constexpr int kSmallLag = C::T::LAG;
    const GemmParams& p = sp.g;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* ring = smem + C::RING_OFF;
    uint8_t* as = smem + C::AS_OFF;
    uint8_t* bs = smem + C::BS_OFF;
    uint8_t* xo = smem + C::XO_OFF;
    float* stg = reinterpret_cast<float*>(smem + C::ST_OFF);
    uint8_t* recv = smem + C::RECV_OFF;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
    uint64_t* x_full = bars;                   // ring slot loaded
    uint64_t* x_emma = x_full + kSmallRing;    // slot released by the Gram MMA (Gram-pass tiles)
    uint64_t* x_eepi = x_emma + kSmallRing;    // slot released by the epilogue (B X tiles: the aX addend)
    uint64_t* d_full = x_eepi + kSmallRing;
    uint64_t* d_empty = d_full + kSmallNB;
    uint64_t* xo_full = d_empty + kSmallNB;    // X' tile written (for the Gram MMA and the store)
    uint64_t* xo_free = xo_full + kSmallXo;    // its Gram MMA done
    uint64_t* xs_done = xo_free + kSmallXo;    // its TMA store has read it
    uint64_t* gram_full = xs_done + kSmallXo;  // A complete in TMEM
    uint64_t* a_ready = gram_full + 1;         // A in shared memory
    uint64_t* aa_full = a_ready + 1;           // AA complete in TMEM
    uint64_t* b_ready = aa_full + 1;           // B in shared memory
    uint64_t* st_done = b_ready + 1;           // an iteration's X' all in global memory
    uint64_t* drain = st_done + 1;
    uint64_t* recv_full = drain + 1;           // CS = 2: the peer's part of this CTA's band of A has arrived
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(recv_full + 1);
    volatile int* bail = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kSmallRing; ++s) {
            mbar_init(smem_u32(&x_full[s]), 1);
            mbar_init(smem_u32(&x_emma[s]), 1);
            mbar_init(smem_u32(&x_eepi[s]), kEpiWarps);
        }
        for (int b = 0; b < kSmallNB; ++b) {
            mbar_init(smem_u32(&d_full[b]), 1);
            mbar_init(smem_u32(&d_empty[b]), kEpiWarps);
        }
        for (int b = 0; b < kSmallXo; ++b) {
            mbar_init(smem_u32(&xo_full[b]), kEpiWarps);
            mbar_init(smem_u32(&xo_free[b]), 1);
            mbar_init(smem_u32(&xs_done[b]), 1);
        }
        mbar_init(smem_u32(gram_full), 1);
        // CS = 2: every lane of the 4 warps that form each half-band of A, in both CTAs
        mbar_init(smem_u32(a_ready), CS == 1 ? kEpiWarps : 2 * 4 * 32);
        mbar_init(smem_u32(recv_full), 4 * 32);
        mbar_init(smem_u32(aa_full), 1);
        mbar_init(smem_u32(b_ready), kEpiWarps);
        mbar_init(smem_u32(st_done), 1);
        mbar_init(smem_u32(drain), 1);
        *bail = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    if constexpr (CS == 2) cluster_sync_all();  // the peer's barriers are initialised before any remote arrive
    else __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t crank = CS == 2 ? (cluster_ctarank() & 1u) : 0u;
    const int cid = static_cast<int>(blockIdx.x) / CS, ncl = static_cast<int>(gridDim.x) / CS;
    // this CTA's tiles of every pass: [tbeg, tbeg + nt) of the unit's np / 64
    const int per = (sp.np / 64 + CS - 1) / CS;
    const int tbeg = static_cast<int>(crank) * per;
    const int nt = min(sp.np / 64, tbeg + per) - tbeg;
    const int S = sp.steps;
    // tile of step t of pass k (k = 0: the Gram pass over X0; k = it + 1: iteration it)
    auto tile_of = [&](int k, int t) { return tbeg + ((sp.reverse && (k & 1)) ? nt - 1 - t : t); };

    if (warp == 0) {
        if (lane == 0) {
            uint32_t kind = 0;              // bit s: slot s last held a B X tile (released by the epilogue)
            uint32_t par_m = 0, par_e = 0;  // bit s: parity of the next release of slot s, per releaser
            uint32_t armed = 0, armed_par = 0;
            int pos = 0, sd = 0;
            bool ok = true;
            for (int u = sp.u0 + cid; u < sp.units && ok; u += ncl) {
                for (int k = 0; k <= S && ok; ++k) {
                    const CUtensorMap* map = (k == 0 || ((k - 1) & 1) == 0) ? &tx0 : &tx1;
                    if (k >= 2) {
                        // X_{k-1} is the previous iteration's X': wait until all of it is stored
                        if (!mbar_wait(smem_u32(st_done), sd & 1, p.err, bail)) { ok = false; break; }
                        ++sd;
                        fence_async_global();
                    }
                    for (int t = 0; t < nt; ++t) {
                        const int s = pos % kSmallRing;
                        if (pos >= kSmallRing) {
                            const bool e = (kind >> s) & 1u;
                            uint32_t& par = e ? par_e : par_m;
                            if (!mbar_wait(smem_u32(e ? &x_eepi[s] : &x_emma[s]), (par >> s) & 1u, p.err, bail)) {
                                ok = false;
                                break;
                            }
                            par ^= 1u << s;
                        }
                        kind = (kind & ~(1u << s)) | ((k > 0 ? 1u : 0u) << s);
                        const uint32_t fb = smem_u32(&x_full[s]);
                        mbar_arrive_expect_tx(fb, kSmallTile);
                        tma_load_3d(smem_u32(ring + s * kSmallTile), map, fb, tile_of(k, t) * 64, 0, u);
                        armed |= 1u << s;
                        armed_par = (armed_par & ~(1u << s)) | ((static_cast<uint32_t>(pos / kSmallRing) & 1u) << s);
                        ++pos;
                    }
                }
            }
            // wait for this CTA's own copies still in flight
            for (int s = 0; s < kSmallRing; ++s)
                if (armed & (1u << s)) mbar_wait(smem_u32(&x_full[s]), (armed_par >> s) & 1u, p.err, bail, false);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t t_a = tmem, t_aa = tmem + 128, t_d = tmem + 256;
            int pos = 0, dpos = 0, xg = 0;
            uint32_t ar = 0, br = 0;
            bool ok = true, first = true;
            // A (+)= T T^T for a 128 x 64 tile T in shared memory
            auto gram_on = [&](uint32_t saddr, bool acc0) {
                const uint64_t d = desc_sw128(saddr);
#pragma unroll
                for (int kk = 0; kk < BK / 16; ++kk) umma_bf16(t_a, d + 2 * kk, d + 2 * kk, C::IDESC_G, (acc0 || kk) ? 1u : 0u);
            };
            for (int u = sp.u0 + cid; u < sp.units && ok; u += ncl) {
                for (int t = 0; t < nt; ++t) {
                    const int s = pos % kSmallRing;
                    if (!mbar_wait(smem_u32(&x_full[s]), (pos / kSmallRing) & 1, p.err, bail)) { ok = false; break; }
                    tc_fence_after();
                    gram_on(smem_u32(ring + s * kSmallTile), t > 0);
                    umma_commit(smem_u32(&x_emma[s]));
                    ++pos;
                }
                if (!ok) break;
                if (!(first && p.inject_no_ready)) umma_commit(smem_u32(gram_full));
                first = false;
                for (int it = 0; it < S && ok; ++it) {
                    if (!(CS == 2 ? mbar_wait_cl(smem_u32(a_ready), ar & 1u, p.err, bail)
                                  : mbar_wait(smem_u32(a_ready), ar & 1u, p.err, bail))) {
                        ok = false;
                        break;
                    }
                    ++ar;
                    tc_fence_after();
                    const uint32_t a0 = smem_u32(as);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint64_t d = desc_sw128(a0 + (kk >> 2) * kSmallTile) + 2 * (kk & 3);
                        umma_bf16(t_aa, d, d, C::IDESC_G, kk ? 1u : 0u);
                    }
                    umma_commit(smem_u32(aa_full));
                    if (!mbar_wait(smem_u32(b_ready), br & 1u, p.err, bail)) { ok = false; break; }
                    ++br;
                    tc_fence_after();
                    const bool last = it + 1 == S;
                    const uint32_t b0 = smem_u32(bs);
                    for (int t = 0; t < nt; ++t) {
                        const int s = pos % kSmallRing;
                        const int db = dpos % kSmallNB;
                        if (!mbar_wait(smem_u32(&x_full[s]), (pos / kSmallRing) & 1, p.err, bail)) { ok = false; break; }
                        if (dpos >= kSmallNB &&
                            !mbar_wait(smem_u32(&d_empty[db]), ((dpos / kSmallNB) - 1) & 1, p.err, bail)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint64_t xd = desc_mn_sw128(smem_u32(ring + s * kSmallTile));
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk)
                            umma_bf16(t_d + 64 * db, desc_sw128(b0 + (kk >> 2) * kSmallTile) + 2 * (kk & 3),
                                      xd + 128 * kk, C::IDESC_BX, kk ? 1u : 0u);
                        umma_commit(smem_u32(&d_full[db]));
                        ++dpos;
                        ++pos;
                        if (!last && t >= kSmallLag) {
                            // the next A from the X' of tile t - kSmallLag: the MMA runs kSmallLag
                            // tiles of B X ahead of the epilogue instead of waiting for it
                            const int b = xg % kSmallXo;
                            if (!mbar_wait(smem_u32(&xo_full[b]), (xg / kSmallXo) & 1, p.err, bail)) { ok = false; break; }
                            tc_fence_after();
                            gram_on(smem_u32(xo + b * kSmallTile), t > kSmallLag);
                            umma_commit(smem_u32(&xo_free[b]));
                            ++xg;
                        }
                    }
                    if (!ok) break;
                    if (!last) {
                        for (int g = nt > kSmallLag ? nt - kSmallLag : 0; g < nt && ok; ++g) {
                            const int b = xg % kSmallXo;
                            if (!mbar_wait(smem_u32(&xo_full[b]), (xg / kSmallXo) & 1, p.err, bail)) { ok = false; break; }
                            tc_fence_after();
                            gram_on(smem_u32(xo + b * kSmallTile), g > 0);
                            umma_commit(smem_u32(&xo_free[b]));
                            ++xg;
                        }
                        if (!ok) break;
                        umma_commit(smem_u32(gram_full));
                    }
                }
            }
            // every MMA this thread issued has completed before TMEM is freed
            umma_commit(smem_u32(drain));
            mbar_wait(smem_u32(drain), 0, p.err, bail, false);
        }
    } else if (warp == 2) {
        if (lane == 0) {
            int xg = 0;
            bool ok = true;
            for (int u = sp.u0 + cid; u < sp.units && ok; u += ncl) {
                for (int it = 0; it + 1 < S && ok; ++it) {
                    const CUtensorMap* map = ((it + 1) & 1) ? &tx1 : &tx0;
                    for (int t = 0; t < nt; ++t) {
                        const int b = xg % kSmallXo;
                        if (!mbar_wait(smem_u32(&xo_full[b]), (xg / kSmallXo) & 1, p.err, bail)) { ok = false; break; }
                        tma_store_3d(map, smem_u32(xo + b * kSmallTile), tile_of(it + 1, t) * 64, 0, u);
                        bulk_commit();
                        bulk_wait_read_all();
                        mbar_arrive(smem_u32(&xs_done[b]));
                        ++xg;
                    }
                    if (!ok) break;
                    bulk_wait_all();
                    fence_async_global();
                    mbar_arrive(smem_u32(st_done));
                }
            }
            bulk_wait_all();
        }
    } else {
        const int ew = warp - 3;         // epilogue warp 0..7
        const int q = warp & 3;          // TMEM lane quadrant of this warp
        const int h = ew >> 2;           // which half of a tile's (or of A's) columns
        const int row = q * 32 + lane;   // row of A, B and X
        float* stage = stg + ew * 1024;
        const uint32_t tl = tmem + (static_cast<uint32_t>(q * 32) << 16);
        int pos = 0, dpos = 0, xg = 0;
        uint32_t gf = 0, af = 0, rf = 0, arc = 0;
        bool ok = true;
        for (int u = sp.u0 + cid; u < sp.units && ok; u += ncl) {
            pos += nt;  // the Gram pass's tiles are released by the MMA
            const float usc = p.unit_scale ? p.unit_scale[u] : 1.f;
            for (int it = 0; it < S && ok; ++it) {
                const bool last = it + 1 == S;
                // A = X X^T (s^2 u u^T in the first iteration), bf16, into shared memory
                ok = mbar_wait(smem_u32(gram_full), gf & 1u, p.err, bail);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                ++gf;
                tc_fence_after();
                const float alpha_t = it == 0 ? 1.f * (usc * usc) : 1.f;
                if constexpr (CS == 1) {
                    uint32_t r0[32], r1[32];
                    tmem_ld32(tl + h * 64, r0);
                    tmem_ld32(tl + h * 64 + 32, r1);
                    tmem_ld_wait();
                    tmem_ld_pin(r0);
                    tmem_ld_pin(r1);
                    uint8_t* dst = as + h * kSmallTile;
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        const uint32_t* r = c < 4 ? r0 + 8 * c : r1 + 8 * (c - 4);
                        *reinterpret_cast<uint4*>(dst + tile_chunk(row, c)) = make_uint4(
                            bf16x2_bits(__uint_as_float(r[0]) * alpha_t, __uint_as_float(r[1]) * alpha_t),
                            bf16x2_bits(__uint_as_float(r[2]) * alpha_t, __uint_as_float(r[3]) * alpha_t),
                            bf16x2_bits(__uint_as_float(r[4]) * alpha_t, __uint_as_float(r[5]) * alpha_t),
                            bf16x2_bits(__uint_as_float(r[6]) * alpha_t, __uint_as_float(r[7]) * alpha_t));
                    }
                    fence_async_smem();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(a_ready));
                } else {
                    // A is the sum of the two CTAs' parts.  CTA r forms rows 64r..64r+63
                    // (TMEM quadrants 2r, 2r+1): the warps of the other two quadrants send
                    // their part of those rows to the peer, the warps of its own two add
                    // the peer's part to theirs, round, and write the band into both CTAs'
                    // A.  Each band is added by one CTA, so both hold the same A.
                    const uint32_t peer = crank ^ 1u;
                    const bool mine = static_cast<uint32_t>(q >> 1) == crank;
                    const int brow = (q & 1) * 32 + lane;  // row inside the band
                    const int sw = lane & 15;              // 16-byte chunk swizzle of the receive rows
                    uint32_t r0[32], r1[32];
                    tmem_ld32(tl + h * 64, r0);
                    tmem_ld32(tl + h * 64 + 32, r1);
                    tmem_ld_wait();
                    tmem_ld_pin(r0);
                    tmem_ld_pin(r1);
                    if (!mine) {
                        const uint32_t rb = mapa_shared(smem_u32(recv + brow * 512 + h * 256), peer);
#pragma unroll
                        for (int c = 0; c < 16; ++c) {
                            const uint32_t* r = c < 8 ? r0 + 4 * c : r1 + 4 * (c - 8);
                            st_cluster_u4(rb + ((c ^ sw) << 4), make_uint4(r[0], r[1], r[2], r[3]));
                        }
                        mbar_arrive_cluster(mapa_shared(smem_u32(recv_full), peer));
                    } else {
                        ok = mbar_wait_cl(smem_u32(recv_full), rf & 1u, p.err, bail);
                        ok = __all_sync(0xffffffffu, ok);
                        if (!ok) break;
                        ++rf;
                        const uint8_t* rb = recv + brow * 512 + h * 256;
                        uint8_t* dst = as + h * kSmallTile;
#pragma unroll
                        for (int c = 0; c < 8; ++c) {
                            const uint32_t* r = c < 4 ? r0 + 8 * c : r1 + 8 * (c - 4);
                            const float4 x0 = *reinterpret_cast<const float4*>(rb + (((2 * c) ^ sw) << 4));
                            const float4 x1 = *reinterpret_cast<const float4*>(rb + (((2 * c + 1) ^ sw) << 4));
                            const float o[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
                            float a8[8];
#pragma unroll
                            for (int e = 0; e < 8; ++e) a8[e] = (__uint_as_float(r[e]) + o[e]) * alpha_t;
                            const uint4 v = make_uint4(bf16x2_bits(a8[0], a8[1]), bf16x2_bits(a8[2], a8[3]),
                                                       bf16x2_bits(a8[4], a8[5]), bf16x2_bits(a8[6], a8[7]));
                            const uint32_t off = static_cast<uint32_t>(h * kSmallTile) + tile_chunk(row, c);
                            *reinterpret_cast<uint4*>(dst + tile_chunk(row, c)) = v;
                            st_cluster_u4(mapa_shared(smem_u32(as) + off, peer), v);
                        }
                        fence_async_smem();
                        fence_async_smem_cluster();
                        mbar_arrive(smem_u32(a_ready));
                        mbar_arrive_cluster(mapa_shared(smem_u32(a_ready), peer));
                    }
                    tc_fence_before();
                    __syncwarp();
                    // the whole of A (half of it written by the peer) before B is formed from it
                    ok = mbar_wait_cl(smem_u32(a_ready), arc & 1u, p.err, bail);
                    ok = __all_sync(0xffffffffu, ok);
                    if (!ok) break;
                    ++arc;
                }
                // B = bA + cAA, bf16, into shared memory
                ok = mbar_wait(smem_u32(aa_full), af & 1u, p.err, bail);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                ++af;
                tc_fence_after();
                {
                    uint32_t r0[32], r1[32];
                    tmem_ld32(tl + 128 + h * 64, r0);
                    tmem_ld32(tl + 128 + h * 64 + 32, r1);
                    tmem_ld_wait();
                    tmem_ld_pin(r0);
                    tmem_ld_pin(r1);
                    const uint8_t* src = as + h * kSmallTile;
                    uint8_t* dst = bs + h * kSmallTile;
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        const uint32_t* r = c < 4 ? r0 + 8 * c : r1 + 8 * (c - 4);
                        float a8[8], o[8];
                        unpack_bf16x8(*reinterpret_cast<const uint4*>(src + tile_chunk(row, c)), a8);
#pragma unroll
                        for (int e = 0; e < 8; ++e) o[e] = fmaf(sp.b, a8[e], __uint_as_float(r[e]) * sp.c);
                        *reinterpret_cast<uint4*>(dst + tile_chunk(row, c)) =
                            make_uint4(bf16x2_bits(o[0], o[1]), bf16x2_bits(o[2], o[3]), bf16x2_bits(o[4], o[5]),
                                       bf16x2_bits(o[6], o[7]));
                    }
                }
                fence_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(b_ready));
                // the last product's destination, once per unit
                NsUnit nu{};
                bool fuse = false;
                int64_t base1 = -1;
                // w buffers of the last pass: the 4 KB of A that this warp wrote (idle
                // once B is formed) and a 4 KB block of the X' tiles, which the last
                // pass does not store
                const uint32_t wbuf0 = smem_u32(as + h * kSmallTile + q * 4096);
                const uint32_t wstep = static_cast<uint32_t>(xo - as);  // buffer 1 - buffer 0
                if (last) {
                    nu = p.ns_units[u];
                    fuse = p.fuse_update && (nu.flags & kNsEpiUpdate);
                    if (fuse && nu.nfrag == 1) base1 = p.frags[nu.frag0].root_off - p.frags[nu.frag0].unit_off;
                }
                if (fuse) {
                    // the X' tiles' last stores have read them
                    for (int k = 1; k <= kSmallXo && k <= xg && ok; ++k)
                        ok = mbar_wait(smem_u32(&xs_done[(xg - k) % kSmallXo]), ((xg - k) / kSmallXo) & 1, p.err, bail);
                    ok = __all_sync(0xffffffffu, ok);
                    if (!ok) break;
                    prefetch_w_chunk(p, nu, base1, q * 32, tile_of(S, 0) * 64 + h * 32, wbuf0);
                    cp_async_commit();
                }
                // the pass over X: X' = a X + B X per tile
                for (int t = 0; t < nt; ++t) {
                    const int j = tile_of(it + 1, t);
                    const int db = dpos % kSmallNB;
                    if (fuse) {
                        if (t + 1 < nt)
                            prefetch_w_chunk(p, nu, base1, q * 32, tile_of(S, t + 1) * 64 + h * 32,
                                             wbuf0 + ((t + 1) & 1) * wstep);
                        cp_async_commit();
                    }
                    ok = mbar_wait(smem_u32(&d_full[db]), (dpos / kSmallNB) & 1, p.err, bail);
                    ok = __all_sync(0xffffffffu, ok);
                    if (!ok) break;
                    tc_fence_after();
                    uint32_t r[32];
                    tmem_ld32(tl + 256 + db * 64 + h * 32, r);
                    tmem_ld_wait();
                    tmem_ld_pin(r);
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&d_empty[db]));
                    ++dpos;
                    // this lane's row of the X tile (32 columns): the aX addend
                    const int s = pos % kSmallRing;
                    ok = mbar_wait(smem_u32(&x_full[s]), (pos / kSmallRing) & 1, p.err, bail);
                    ok = __all_sync(0xffffffffu, ok);
                    if (!ok) break;
                    const uint8_t* xt = ring + s * kSmallTile;
                    float y[32];
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        float x8[8];
                        unpack_bf16x8(*reinterpret_cast<const uint4*>(xt + tile_chunk(row, 4 * h + c)), x8);
#pragma unroll
                        for (int e = 0; e < 8; ++e) y[8 * c + e] = fmaf(sp.a, x8[e], __uint_as_float(r[8 * c + e]));
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&x_eepi[s]));
                    ++pos;
                    if (it == 0) {
#pragma unroll
                        for (int e = 0; e < 32; ++e) y[e] *= usc;
                    }
                    if (!last) {
                        // bf16 X' into its shared tile, for the next A and the store
                        const int b = xg % kSmallXo;
                        if (xg >= kSmallXo) {
                            ok = mbar_wait(smem_u32(&xo_free[b]), ((xg / kSmallXo) - 1) & 1, p.err, bail) &&
                                 mbar_wait(smem_u32(&xs_done[b]), ((xg / kSmallXo) - 1) & 1, p.err, bail);
                            ok = __all_sync(0xffffffffu, ok);
                            if (!ok) break;
                        }
                        uint8_t* dst = xo + b * kSmallTile;
#pragma unroll
                        for (int c = 0; c < 4; ++c)
                            *reinterpret_cast<uint4*>(dst + tile_chunk(row, 4 * h + c)) =
                                make_uint4(bf16x2_bits(y[8 * c], y[8 * c + 1]), bf16x2_bits(y[8 * c + 2], y[8 * c + 3]),
                                           bf16x2_bits(y[8 * c + 4], y[8 * c + 5]),
                                           bf16x2_bits(y[8 * c + 6], y[8 * c + 7]));
                        fence_async_smem();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(smem_u32(&xo_full[b]));
                        ++xg;
                    } else {
                        // v = a X + B X: this lane's row into the warp's staging tile, then
                        // v stored or f2 and G applied, as in the three-launch form
#pragma unroll
                        for (int c4 = 0; c4 < 8; ++c4)
                            *stage4(stage, lane, c4) = make_float4(y[4 * c4], y[4 * c4 + 1], y[4 * c4 + 2], y[4 * c4 + 3]);
                        __syncwarp();
                        if (fuse) {
                            cp_async_wait_1();  // this tile's w (the next tile's may be in flight)
                            final_update_chunk_buf<kSmallWGroup>(p, nu, base1, stage, q * 32, j * 64 + h * 32,
                                                   reinterpret_cast<const float4*>(as + h * kSmallTile + q * 4096 +
                                                                                   (t & 1) * wstep));
                        } else {
                            store_final_chunk(p, nu, fuse, base1, stage, row, q * 32, j * 64 + h * 32);
                        }
                        __syncwarp();
                    }
                }
                if (fuse) cp_async_wait_all();
            }
        }
        cp_async_wait_all();
    }
    if constexpr (CS == 2) {
        // the peer may still write this CTA's shared memory or arrive on its
        // barriers: both CTAs stay until every role of both is done
        __syncwarp();
        tc_fence_before();
        cluster_sync_all();
    } else {
        __syncthreads();
    }
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

template <int CS>
cudaError_t launch_small_cs(const CUtensorMap& x0, const CUtensorMap& x1, const SmallNsParams& sp, cudaStream_t st) {
    using C = SmallCfg<CS>;
    static bool configured[64] = {false};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !configured[dev]) {
        cudaError_t e = cudaFuncSetAttribute(ns_small_kernel<CS>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (e != cudaSuccess) return e;
        configured[dev] = true;
    }
    const int cap = device_sm_count() / CS;
    const int nu = sp.units - sp.u0;
    const int clusters = nu < cap ? nu : cap;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(CS * clusters, 1, 1);
    cfg.blockDim = dim3(kSmallThreads, 1, 1);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CS;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = CS == 2 ? 1 : 0;
    note_launch();
    return cudaLaunchKernelEx(&cfg, ns_small_kernel<CS>, x0, x1, sp);
}

// A class with at most one unit per CTA pair splits each unit over a pair
// (when its units have at least two tiles per pass); otherwise one CTA per
// unit, in whole rounds of one unit per SM, and the units of a last, partial
// round split over pairs (half as long: 960 Video-DiT heads on 152 SMs run 6
// rounds and then 48 units on 48 pairs, 3.65 instead of 3.82 ms).
cudaError_t launch_small(const CUtensorMap& x0, const CUtensorMap& x1, const SmallNsParams& sp0, cudaStream_t st) {
    if (sp0.units == 0) return cudaSuccess;
    SmallNsParams sp = sp0;
    sp.u0 = 0;
    const int sms = device_sm_count();
    const bool splittable = sp.np / 64 >= 2;
    if (splittable && 2 * sp.units <= sms) return launch_small_cs<2>(x0, x1, sp, st);
    const int whole = sp.units / sms * sms;  // units in whole rounds
    if (!splittable || whole == 0 || whole == sp.units) return launch_small_cs<1>(x0, x1, sp, st);
    SmallNsParams rounds = sp, tail = sp;
    rounds.units = whole;
    tail.u0 = whole;
    cudaError_t e = launch_small_cs<1>(x0, x1, rounds, st);
    return e != cudaSuccess ? e : launch_small_cs<2>(x0, x1, tail, st);
}

template <bool B_MN>
cudaError_t launch_gemm_pair(const CUtensorMap& tma, const CUtensorMap& tmb, const GemmParams& p0, cudaStream_t st) {
    using C = PairCfg<B_MN>;
    static bool configured[64] = {false};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !configured[dev]) {
        cudaError_t e = cudaFuncSetAttribute(ns_gemm_pair_kernel<B_MN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             C::SMEM);
        if (e != cudaSuccess) return e;
        configured[dev] = true;
    }
    GemmParams p = p0;
    p.tiles_m = (p.M + 255) / 256;
    p.tiles_n = (p.N + C::BNP - 1) / C::BNP;
    p.num_kb = (p.K + BK - 1) / BK;
    const int total = p.units * (p.tile_tab ? p.tab_len : p.tiles_m * p.tiles_n);
    if (total == 0) return cudaSuccess;
    const int pairs = total < device_sm_count() / 2 ? total : device_sm_count() / 2;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * pairs, 1, 1);
    cfg.blockDim = dim3(kGemmThreads, 1, 1);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    note_launch();
    return cudaLaunchKernelEx(&cfg, ns_gemm_pair_kernel<B_MN>, tma, tmb, p);
}

template <int BN, bool B_MN>
cudaError_t launch_gemm_bn(const CUtensorMap& tma, const CUtensorMap& tmb, const GemmParams& p0, cudaStream_t st) {
    using C = GemmCfg<BN, B_MN>;
    static bool configured[64] = {false};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !configured[dev]) {
        cudaError_t e = cudaFuncSetAttribute(ns_gemm_kernel<BN, B_MN>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (e != cudaSuccess) return e;
        configured[dev] = true;
    }
    GemmParams p = p0;
    p.tiles_m = (p.M + BM - 1) / BM;
    p.tiles_n = (p.N + BN - 1) / BN;
    p.num_kb = (p.K + BK - 1) / BK;
    const int total = p.units * (p.tile_tab ? p.tab_len : p.tiles_m * p.tiles_n);
    if (total == 0) return cudaSuccess;
    const int grid = total < device_sm_count() ? total : device_sm_count();
    note_launch();
    ns_gemm_kernel<BN, B_MN><<<grid, kGemmThreads, C::SMEM, st>>>(tma, tmb, p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_ns_prepare(const NsClassDev& c, const NsUnit* units_dev, const uint16_t* u_root,
                              const uint16_t* u_stage, char* ws, cudaStream_t st) {
    dim3 g(c.np / 64, c.mp / 64, c.n_units);
    note_launch();
    ns_prepare_kernel<<<g, kPrepThreads, 0, st>>>(units_dev, u_root, u_stage, reinterpret_cast<float*>(ws + c.part_off),
                                                  reinterpret_cast<uint16_t*>(ws + c.x_off[0]), c.m, c.n, c.np);
    return cudaGetLastError();
}

cudaError_t launch_ns_f0_prepare(const NsClassDev& c, const NsUnit* units_dev, const NsFrag* frags_dev, float* m,
                                 const float* g, float mu, int nesterov, char* ws, cudaStream_t st) {
    dim3 grid(c.np / 64, c.mp / 64, c.n_units);
    note_launch();
    f0_prepare_kernel<<<grid, kPrepThreads, 0, st>>>(units_dev, frags_dev, m, g, mu, nesterov,
                                                     reinterpret_cast<float*>(ws + c.part_off),
                                                     reinterpret_cast<uint16_t*>(ws + c.x_off[0]), c.m, c.n, c.np);
    return cudaGetLastError();
}

cudaError_t launch_ns_norm(const NsClassDev& c, char* ws, float eps, cudaStream_t st) {
    note_launch();
    ns_norm_final_kernel<<<c.n_units, kNormThreads, 0, st>>>(reinterpret_cast<const float*>(ws + c.part_off), c.parts,
                                                             reinterpret_cast<float*>(ws + c.inv_off), eps);
    return cudaGetLastError();
}

cudaError_t launch_ns_small(const CUtensorMap& x0, const CUtensorMap& x1, const SmallNsParams& p, cudaStream_t st) {
    return launch_small(x0, x1, p, st);
}

cudaError_t launch_ns_gemm_pair(const CUtensorMap& tma, const CUtensorMap& tmb, const GemmParams& p, int b_mn,
                                cudaStream_t st) {
    return b_mn ? launch_gemm_pair<true>(tma, tmb, p, st) : launch_gemm_pair<false>(tma, tmb, p, st);
}

cudaError_t launch_ns_gemm(const CUtensorMap& tma, const CUtensorMap& tmb, const GemmParams& p, int bn, int b_mn,
                           cudaStream_t st) {
    if (b_mn) return bn == 256 ? launch_gemm_bn<256, true>(tma, tmb, p, st) : launch_gemm_bn<128, true>(tma, tmb, p, st);
    return bn == 256 ? launch_gemm_bn<256, false>(tma, tmb, p, st) : launch_gemm_bn<128, false>(tma, tmb, p, st);
}

}  // namespace hm
