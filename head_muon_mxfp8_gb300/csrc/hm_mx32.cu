// G with 32 x 32 MX blocks over the emulated rank segments, and Tw's scale
// relayout into the 128 x 4 tiled layout of block-scaled GEMMs.
//
// SS-HSDP section 3.1 example EG1: G uses 32 x 32 block quantization in a
// k-major layout; Tw relays the scales out for the GEMM kernel; section 4.1:
// scale-layout transforms are batched across tensors.
#include "hm.h"
#include "hm_internal.h"
#include "hm_mx_device.cuh"

#include <cstring>

namespace hm {

namespace {

__device__ __forceinline__ int64_t logical_to_root(const ChainArgs& ch, int64_t x) {
    if (ch.so == 0) return x;
    int lo = 0, hi = ch.so - 1;  // last chunk c with edges[c] <= x (empty chunks skipped)
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (ch.edges[mid] <= x) lo = mid;
        else hi = mid - 1;
    }
    return ch.chunk_base[lo] + (x - ch.edges[lo]);
}

// One warp per 32 x 32 block: lane l owns column l of the block, the warp walks
// its 32 rows (each row is 32 consecutive logical elements, one segment).
__global__ void __launch_bounds__(256) requant_32x32_kernel(const __grid_constant__ ChainArgs ch,
                                                             const __grid_constant__ Mx32Args ta,
                                                             const float* __restrict__ w, uint8_t* __restrict__ q,
                                                             uint8_t* __restrict__ scales) {
    const int lane = threadIdx.x & 31;
    const int64_t total = ta.block_prefix[ta.n];
    const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
    for (int64_t b = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); b < total;
         b += warps) {
        int t = 0;
        while (ta.block_prefix[t + 1] <= b) ++t;
        const int64_t k = ta.k[t];
        const int64_t kb = k >> 5;
        const int64_t local = b - ta.block_prefix[t];
        const int64_t br = local / kb, bc = local - br * kb;
        const int64_t row0 = ta.src[t] + (br * 32) * k + bc * 32;
        int64_t root[32];
        float x[32];
        float amax = 0.f;
#pragma unroll
        for (int r = 0; r < 32; ++r) {
            root[r] = logical_to_root(ch, row0 + r * k) + lane;
            x[r] = __ldg(w + root[r]);
            amax = fmaxf(amax, fabsf(x[r]));
        }
#pragma unroll
        for (int sh = 16; sh; sh >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, sh));
        const int e = mx_scale_exponent(amax);
        const float sc = mx_inv_scale(e);
#pragma unroll
        for (int r = 0; r < 32; r += 2) {
            const uint16_t c2 = cvt_e4m3x2(x[r] * sc, x[r + 1] * sc);
            q[root[r]] = static_cast<uint8_t>(c2 & 0xFFu);
            q[root[r + 1]] = static_cast<uint8_t>(c2 >> 8);
        }
        if (lane == 0) scales[ta.scale_off[t] + local] = static_cast<uint8_t>(e + 127);
    }
}

__global__ void __launch_bounds__(256) scale_relayout_kernel(const __grid_constant__ RelayoutArgs ra,
                                                              const uint8_t* __restrict__ src,
                                                              uint8_t* __restrict__ dst) {
    const int64_t total = ra.out_prefix[ra.n];
    for (int64_t o = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; o < total;
         o += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        int t = 0;
        while (ra.out_prefix[t + 1] <= o) ++t;
        const int64_t local = o - ra.out_prefix[t];
        const int64_t ct = (ra.kb[t] + 3) >> 2;
        const int64_t tile = local >> 9;
        const int within = static_cast<int>(local & 511);
        const int64_t r = (tile / ct) * 128 + ((within & 15) >> 2) * 32 + (within >> 4);
        const int64_t c = (tile % ct) * 4 + (within & 3);
        uint8_t val = 0;
        if (r < ra.rows[t] && c < ra.kb[t]) val = src[ra.src[t] + (r / ra.block_rows[t]) * ra.kb[t] + c];
        dst[ra.dst[t] + local] = val;
    }
}

}  // namespace

cudaError_t launch_requant_32x32(const ChainArgs& ch, const Mx32Args& ta, const float* w, uint8_t* q,
                                 uint8_t* scales, cudaStream_t st) {
    const int64_t total = ta.block_prefix[ta.n];
    if (total == 0) return cudaSuccess;
    int64_t blocks = (total + 7) / 8;
    const int64_t cap = static_cast<int64_t>(device_sm_count()) * 16;
    if (blocks > cap) blocks = cap;
    requant_32x32_kernel<<<static_cast<int>(blocks), 256, 0, st>>>(ch, ta, w, q, scales);
    return cudaGetLastError();
}

cudaError_t launch_scale_relayout(const RelayoutArgs& ra, const uint8_t* src, uint8_t* dst, cudaStream_t st) {
    const int64_t total = ra.out_prefix[ra.n];
    if (total == 0) return cudaSuccess;
    int64_t blocks = (total + 255) / 256;
    const int64_t cap = static_cast<int64_t>(device_sm_count()) * 16;
    if (blocks > cap) blocks = cap;
    scale_relayout_kernel<<<static_cast<int>(blocks), 256, 0, st>>>(ra, src, dst);
    return cudaGetLastError();
}

}  // namespace hm
