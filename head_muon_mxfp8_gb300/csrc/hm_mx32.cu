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

// One warp per strip of 32 rows x 128 columns (four 32 x 32 blocks): lane l
// owns columns 4l .. 4l+3, i.e. eight lanes per block; every row of a block is
// 32 consecutive logical elements, so the four columns of a lane always sit in
// one rank segment.  Loads are 16 bytes per lane, codes are stored 4 per lane.
__device__ __forceinline__ int64_t walk_to_root(const ChainArgs& ch, int& c, int64_t x) {
    if (ch.so == 0) return x;
    while (c + 1 < ch.so && ch.edges[c + 1] <= x) ++c;
    return ch.chunk_base[c] + (x - ch.edges[c]);
}

__global__ void __launch_bounds__(128) requant_32x32_kernel(const __grid_constant__ ChainArgs ch,
                                                             const __grid_constant__ Mx32Args ta,
                                                             const float* __restrict__ w, uint8_t* __restrict__ q,
                                                             uint8_t* __restrict__ scales) {
    const int lane = threadIdx.x & 31;
    const int64_t total = ta.block_prefix[ta.n];  // counted in strips here
    const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
    for (int64_t b = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); b < total;
         b += warps) {
        int t = 0;
        while (ta.block_prefix[t + 1] <= b) ++t;
        const int64_t k = ta.k[t];
        const int64_t strips = (k + 127) >> 7;
        const int64_t local = b - ta.block_prefix[t];
        const int64_t br = local / strips, st = local - br * strips;
        const int64_t col = st * 128 + lane * 4;
        const bool live = col < k;  // uniform over the 8 lanes of a block
        const int64_t x0 = ta.src[t] + (br * 32) * k + col;
        int c = 0;
        if (ch.so) {  // chunk holding the first row: binary search, then walk forward
            int lo = 0, hi = ch.so - 1;
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (ch.edges[mid] <= x0) lo = mid;
                else hi = mid - 1;
            }
            c = lo;
        }
        float4 x[32];
        float amax = 0.f;
#pragma unroll
        for (int r = 0; r < 32; ++r) {
            x[r] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (live) x[r] = __ldg(reinterpret_cast<const float4*>(w + walk_to_root(ch, c, x0 + r * k)));
            amax = fmaxf(amax, fmaxf(fmaxf(fabsf(x[r].x), fabsf(x[r].y)), fmaxf(fabsf(x[r].z), fabsf(x[r].w))));
        }
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 4));
        if (!live) continue;
        const int e = mx_scale_exponent(amax);
        const float sc = mx_inv_scale(e);
        int c2 = 0;
        if (ch.so) {
            int lo = 0, hi = ch.so - 1;
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (ch.edges[mid] <= x0) lo = mid;
                else hi = mid - 1;
            }
            c2 = lo;
        }
#pragma unroll
        for (int r = 0; r < 32; ++r) {
            const uint32_t code = cvt_e4m3x2(x[r].x * sc, x[r].y * sc) |
                                  (static_cast<uint32_t>(cvt_e4m3x2(x[r].z * sc, x[r].w * sc)) << 16);
            *reinterpret_cast<uint32_t*>(q + walk_to_root(ch, c2, x0 + r * k)) = code;
        }
        if ((lane & 7) == 0) scales[ta.scale_off[t] + br * (k >> 5) + (col >> 5)] = static_cast<uint8_t>(e + 127);
    }
}

// Each thread writes one 16-byte group of a tile: rows l, l+32, l+64, l+96
// (l = group index within the tile) x 4 scale columns.
__global__ void __launch_bounds__(256) scale_relayout_kernel(const __grid_constant__ RelayoutArgs ra,
                                                              const uint8_t* __restrict__ src,
                                                              uint8_t* __restrict__ dst) {
    const int64_t total = ra.out_prefix[ra.n] >> 4;
    for (int64_t o = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; o < total;
         o += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        int t = 0;
        while ((ra.out_prefix[t + 1] >> 4) <= o) ++t;
        const int64_t local = o - (ra.out_prefix[t] >> 4);  // 16-byte group index in this item
        const int64_t ct = (ra.kb[t] + 3) >> 2;
        const int64_t tile = local >> 5;
        const int l = static_cast<int>(local & 31);
        const int64_t r0 = (tile / ct) * 128 + l;
        const int64_t c0 = (tile % ct) * 4;
        uint32_t word[4];
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
            const int64_t r = r0 + 32 * q4;
            uint32_t v = 0;
#pragma unroll
            for (int c = 0; c < 4; ++c)
                if (r < ra.rows[t] && c0 + c < ra.kb[t])
                    v |= static_cast<uint32_t>(src[ra.src[t] + (r / ra.block_rows[t]) * ra.kb[t] + c0 + c]) << (8 * c);
            word[q4] = v;
        }
        uint8_t* out = dst + ra.dst[t] + local * 16;
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
#pragma unroll
            for (int c = 0; c < 4; ++c) out[q4 * 4 + c] = static_cast<uint8_t>(word[q4] >> (8 * c));
        }
    }
}

}  // namespace

cudaError_t launch_requant_32x32(const ChainArgs& ch, const Mx32Args& ta, const float* w, uint8_t* q,
                                 uint8_t* scales, cudaStream_t st) {
    const int64_t total = ta.block_prefix[ta.n];
    if (total == 0) return cudaSuccess;
    const int64_t blocks = (total + 3) / 4;
    note_launch();
    requant_32x32_kernel<<<resident_grid(requant_32x32_kernel, 128, blocks), 128, 0, st>>>(ch, ta, w, q, scales);
    return cudaGetLastError();
}

cudaError_t launch_scale_relayout(const RelayoutArgs& ra, const uint8_t* src, uint8_t* dst, cudaStream_t st) {
    const int64_t total = ra.out_prefix[ra.n];
    if (total == 0) return cudaSuccess;
    const int64_t blocks = (total / 16 + 255) / 256;
    note_launch();
    scale_relayout_kernel<<<resident_grid(scale_relayout_kernel, 256, blocks), 256, 0, st>>>(ra, src, dst);
    return cudaGetLastError();
}

}  // namespace hm
