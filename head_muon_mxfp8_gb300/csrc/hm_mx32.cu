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
        // chunk holding the first row (binary search); when all 32 rows lie in
        // it -- the usual case, chunks are millions of elements -- the rows'
        // root addresses are affine and all 32 loads issue back to back
        int c = 0;
        int64_t rb = 0;  // root offset minus logical offset inside chunk c
        bool affine = true;
        if (ch.so) {
            int lo = 0, hi = ch.so - 1;
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (ch.edges[mid] <= x0) lo = mid;
                else hi = mid - 1;
            }
            c = lo;
            rb = ch.chunk_base[c] - ch.edges[c];
            affine = c + 1 >= ch.so || x0 + 31 * k < ch.edges[c + 1];
        }
        float4 x[32];
        if (!live) {
#pragma unroll
            for (int r = 0; r < 32; ++r) x[r] = make_float4(0.f, 0.f, 0.f, 0.f);
        } else if (affine) {
            const float* src = w + rb + x0;
#pragma unroll
            for (int r = 0; r < 32; ++r) x[r] = __ldg(reinterpret_cast<const float4*>(src + r * k));
        } else {
            int cw = c;
#pragma unroll
            for (int r = 0; r < 32; ++r) x[r] = __ldg(reinterpret_cast<const float4*>(w + walk_to_root(ch, cw, x0 + r * k)));
        }
        float amax = 0.f;
#pragma unroll
        for (int r = 0; r < 32; ++r)
            amax = fmaxf(amax, fmaxf(fmaxf(fabsf(x[r].x), fabsf(x[r].y)), fmaxf(fabsf(x[r].z), fabsf(x[r].w))));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 4));
        if (!live) continue;
        const int e = mx_scale_exponent(amax);
        const float sc = mx_inv_scale(e);
        int cw = c;
#pragma unroll
        for (int r = 0; r < 32; ++r) {
            const uint32_t code = cvt_e4m3x2(x[r].x * sc, x[r].y * sc) |
                                  (static_cast<uint32_t>(cvt_e4m3x2(x[r].z * sc, x[r].w * sc)) << 16);
            const int64_t o = affine ? rb + x0 + r * k : walk_to_root(ch, cw, x0 + r * k);
            *reinterpret_cast<uint32_t*>(q + o) = code;
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
        const int64_t kb = ra.kb[t];
        // 4-byte source words when every scale row starts 4-byte aligned and
        // the tile's 4 columns are all inside the row
        const bool words = (ra.flags[t] & kRelayoutSrcWords) && c0 + 4 <= kb;
        uint32_t word[4];
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
            const int64_t r = r0 + 32 * q4;
            uint32_t v = 0;
            if (r < ra.rows[t]) {
                const uint8_t* row = src + ra.src[t] + (r / ra.block_rows[t]) * kb;
                if (words) {
                    v = __ldg(reinterpret_cast<const uint32_t*>(row + c0));
                } else {
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        if (c0 + c < kb) v |= static_cast<uint32_t>(row[c0 + c]) << (8 * c);
                }
            }
            word[q4] = v;
        }
        uint8_t* out = dst + ra.dst[t] + local * 16;
        if (ra.flags[t] & kRelayoutDst16) {
            *reinterpret_cast<uint4*>(out) = make_uint4(word[0], word[1], word[2], word[3]);
        } else {
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
#pragma unroll
                for (int c = 0; c < 4; ++c) out[q4 * 4 + c] = static_cast<uint8_t>(word[q4] >> (8 * c));
            }
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
