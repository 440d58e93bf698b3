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

// Work units of 128 scale rows x 160 scale columns (forty 128 x 4 tiles side
// by side).  The 256 threads read the unit's rows as 16-byte pieces (five per
// thread, all in flight; a 160-byte row is a whole scale row of a K = 5120
// tensor, so the unit is one contiguous 20 KB block) into shared memory,
// then write one 16-byte group each of the forty tiles -- rows l, l+32,
// l+64, l+96 of a tile (l = group index) x its 4 scale columns -- so the
// unit leaves as 20 KB of contiguous stores.
constexpr int kRelayoutCols = 160;                      // scale columns per work unit
constexpr int kRelayoutTiles = kRelayoutCols / 4;       // 40 tiles
constexpr int kRelayoutRowWords = kRelayoutCols / 4 + 1;  // 41: odd stride, conflict-free column reads
constexpr int kRelayoutPieces = 128 * kRelayoutCols / 16 / 256;  // 16-byte loads per thread: 5

__global__ void __launch_bounds__(256) scale_relayout_kernel(const __grid_constant__ RelayoutArgs ra,
                                                              const uint8_t* __restrict__ src,
                                                              uint8_t* __restrict__ dst) {
    __shared__ uint32_t S[128 * kRelayoutRowWords];
    const int tid = threadIdx.x;
    const int64_t total = ra.work_prefix[ra.n];
    for (int64_t wu = blockIdx.x; wu < total; wu += gridDim.x) {
        int lo = 0, hi = ra.n - 1;  // the item holding work unit wu
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (ra.work_prefix[mid] <= wu) lo = mid;
            else hi = mid - 1;
        }
        const int t = lo;
        const int64_t local = wu - ra.work_prefix[t];
        const int64_t kb = ra.kb[t];
        const int64_t ct = (kb + 3) >> 2;                                 // tiles across
        const int64_t groups = (ct + kRelayoutTiles - 1) / kRelayoutTiles;  // work units across
        const int64_t band = local / groups, J = local - band * groups;
        const bool vec = (ra.flags[t] & kRelayoutSrc16) != 0;
        // load: piece p -> row p / 10, 16 bytes from column 160 J + 16 (p % 10)
        uint32_t wv[kRelayoutPieces][4];
#pragma unroll
        for (int k = 0; k < kRelayoutPieces; ++k) {
            const int piece = tid + k * 256;
            const int rr = piece / 10, part = piece % 10;
            const int64_t r = band * 128 + rr;
            const int64_t c0 = J * kRelayoutCols + part * 16;
            wv[k][0] = wv[k][1] = wv[k][2] = wv[k][3] = 0u;
            if (r < ra.rows[t] && c0 < kb) {
                const uint8_t* row = src + ra.src[t] + (r / ra.block_rows[t]) * kb + c0;
                if (vec && c0 + 16 <= kb) {
                    const uint4 x = __ldg(reinterpret_cast<const uint4*>(row));
                    wv[k][0] = x.x; wv[k][1] = x.y; wv[k][2] = x.z; wv[k][3] = x.w;
                } else {
#pragma unroll
                    for (int c = 0; c < 16; ++c)
                        if (c0 + c < kb) wv[k][c >> 2] |= static_cast<uint32_t>(row[c]) << (8 * (c & 3));
                }
            }
        }
#pragma unroll
        for (int k = 0; k < kRelayoutPieces; ++k) {
            const int piece = tid + k * 256;
            const int rr = piece / 10, part = piece % 10;
#pragma unroll
            for (int e = 0; e < 4; ++e) S[rr * kRelayoutRowWords + part * 4 + e] = wv[k][e];
        }
        __syncthreads();
        // store: group g -> tile g / 32 of the forty, group l = g % 32 in it
        uint8_t* out0 = dst + ra.dst[t] + (band * ct + J * kRelayoutTiles) * 512;
        const bool dvec = (ra.flags[t] & kRelayoutDst16) != 0;
#pragma unroll
        for (int k = 0; k < kRelayoutPieces; ++k) {
            const int g = tid + k * 256;
            const int jj = g >> 5, l = g & 31;
            if (J * kRelayoutTiles + jj >= ct) continue;
            uint32_t word[4];
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) word[q4] = S[(l + 32 * q4) * kRelayoutRowWords + jj];
            uint8_t* out = out0 + g * 16;
            if (dvec) {
                *reinterpret_cast<uint4*>(out) = make_uint4(word[0], word[1], word[2], word[3]);
            } else {
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
#pragma unroll
                    for (int c = 0; c < 4; ++c) out[q4 * 4 + c] = static_cast<uint8_t>(word[q4] >> (8 * c));
                }
            }
        }
        __syncthreads();
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
    const int64_t total = ra.work_prefix[ra.n];
    if (total == 0) return cudaSuccess;
    note_launch();
    scale_relayout_kernel<<<resident_grid(scale_relayout_kernel, 256, total), 256, 0, st>>>(ra, src, dst);
    return cudaGetLastError();
}

}  // namespace hm
