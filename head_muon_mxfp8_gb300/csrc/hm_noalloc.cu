// Newton-Schulz of one update unit with no device allocation at all.
//
// For callers that cannot call cudaMalloc: code inside a framework that has
// already handed all device memory to its own caching allocator (an
// allocation of its own would fail or fragment that pool), and
// latency-critical paths that must not take the driver's allocation lock or
// an implicit device synchronisation.  The caller passes u and v; every intermediate (X,
// A, B, the norm partials and the unit descriptor) lives in one file-scope
// __device__ array of fixed size, which every GPU that loads the library
// holds until the process exits.
//
// The computation is the same as the Newton-Schulz stage of
// muon_update_units: the same norm, prepare and tcgen05 GEMM kernels, on the
// built-in scratch instead of a caller workspace.
#include "hm.h"
#include "hm_internal.h"

#include <mutex>

namespace {

constexpr int kMaxM = HM_NOALLOC_MAX_MIN_DIM;   // padded Gram size of the scratch
constexpr int kMaxN = HM_NOALLOC_MAX_MAX_DIM;
constexpr size_t kSlot = 1024;
constexpr size_t kXBytes = static_cast<size_t>(kMaxM) * kMaxN * 2;
constexpr size_t kABytes = static_cast<size_t>(kMaxM) * kMaxM * 2;
// one norm partial per 64 x 64 tile of X
constexpr size_t kPartsBytes = (static_cast<size_t>(kMaxM / 64) * (kMaxN / 64) * 4 + kSlot - 1) / kSlot * kSlot;
// layout: unit descriptor | X0 | X1 | A | B | partials | 1/norm
constexpr size_t kOffUnit = 0;
constexpr size_t kOffX0 = kSlot;
constexpr size_t kOffX1 = kOffX0 + kXBytes;
constexpr size_t kOffA = kOffX1 + kXBytes;
constexpr size_t kOffB = kOffA + kABytes;
constexpr size_t kOffParts = kOffB + kABytes;
constexpr size_t kOffInv = kOffParts + kPartsBytes;
constexpr size_t kScratchBytes = kOffInv + kSlot;
static_assert(kScratchBytes == HM_NOALLOC_SCRATCH_BYTES, "scratch size stated in hm.h");

static __device__ __align__(256) unsigned char g_ns_scratch[kScratchBytes];

__global__ void write_unit_kernel(hm::NsUnit* dst, hm::NsUnit unit) { *dst = unit; }

// Device address of the scratch array on the current device, looked up once
// per device (the array's host-side name is not a device address).
char* scratch_on_current_device() {
    static std::mutex mu;
    static char* cached[64] = {nullptr};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lk(mu);
    if (!cached[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_ns_scratch) != cudaSuccess) return nullptr;
        cached[dev] = static_cast<char*>(p);
    }
    return cached[dev];
}

bool device_is_sm103() {
    int dev = 0, major = 0, minor = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return false;
    return major == 10 && minor == 3;
}

using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn encoder() {
    static EncodeFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeFn>(f);
    });
    return fn;
}

// [1][rows][inner] bf16, box [1][box_rows][64], 128-byte swizzle.
bool map_bf16(CUtensorMap* m, void* base, int64_t inner, int64_t rows, int box_rows) {
    EncodeFn fn = encoder();
    if (!fn) return false;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows), 1};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(inner * 2), static_cast<cuuint64_t>(inner * rows * 2)};
    cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_rows), 1};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

extern "C" hm_status newton_schulz_noalloc(const uint16_t* u, int32_t rows, int32_t cols, float* v,
                                           const hm_muon_hparams* hp, void* stream) {
    if (!u || !v || !hp || rows < 1 || cols < 1 || hp->ns_steps < 1 || hp->ns_steps > 100) return HM_ERR_ARG;
    const int m = rows < cols ? rows : cols;
    const int n = rows < cols ? cols : rows;
    if (m > kMaxM || n > kMaxN) return HM_ERR_WORKSPACE;  // larger than the built-in scratch
    if ((static_cast<int64_t>(rows) * cols) % 8 || (reinterpret_cast<uintptr_t>(u) & 15u) ||
        (reinterpret_cast<uintptr_t>(v) & 3u))
        return HM_ERR_ALIGN;
    if (!device_is_sm103()) return HM_ERR_ARCH;
    char* ws = scratch_on_current_device();
    if (!ws) return HM_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);

    hm::NsUnit unit{};
    unit.rows = rows;
    unit.cols = cols;
    unit.flags = rows > cols ? hm::kNsTransposed : 0;
    hm::NsClassDev c{};
    c.m = m;
    c.n = n;
    c.mp = kMaxM;
    c.np = (n + 63) / 64 * 64;
    c.n_units = 1;
    c.parts = (c.np / 64) * (c.mp / 64);
    c.x_off[0] = kOffX0;
    c.x_off[1] = kOffX1;
    c.a_off = kOffA;
    c.b_off = kOffB;
    c.part_off = kOffParts;
    c.inv_off = kOffInv;
    hm::NsUnit* unit_dev = reinterpret_cast<hm::NsUnit*>(ws + kOffUnit);

    CUtensorMap x_map[2], x_mn[2], a_map, b_map;
    const int bn3 = c.np >= 256 ? 256 : 128;
    bool ok = true;
    for (int b = 0; b < 2; ++b) {
        ok = ok && map_bf16(&x_map[b], ws + c.x_off[b], c.np, c.mp, 128);
        ok = ok && map_bf16(&x_mn[b], ws + c.x_off[b], c.np, c.mp, 64);
    }
    ok = ok && map_bf16(&a_map, ws + c.a_off, c.mp, c.mp, 128);
    ok = ok && map_bf16(&b_map, ws + c.b_off, c.mp, c.mp, 128);
    if (!ok) return HM_ERR_CUDA;

    hm::note_launch();
    write_unit_kernel<<<1, 1, 0, st>>>(unit_dev, unit);
    if (cudaGetLastError() != cudaSuccess) return HM_ERR_CUDA;
    if (hm::launch_ns_prepare(c, unit_dev, u, nullptr, ws, st) != cudaSuccess ||
        hm::launch_ns_norm(c, ws, hp->eps, st) != cudaSuccess)
        return HM_ERR_CUDA;
    const float* inv = reinterpret_cast<const float*>(ws + c.inv_off);
    auto bf = [&](size_t off) { return reinterpret_cast<uint16_t*>(ws + off); };
    int cur = 0;
    for (int it = 0; it < hp->ns_steps; ++it) {
        hm::GemmParams g1{};
        g1.M = c.mp; g1.N = c.mp; g1.K = c.np; g1.units = 1;
        g1.epi = hm::kEpiGram; g1.alpha = 1.f; g1.beta = 0.f;
        g1.out = bf(c.a_off); g1.out_us = static_cast<int64_t>(c.mp) * c.mp; g1.ld_out = c.mp;
        g1.err = hm::device_error_word();
        g1.unit_scale = it == 0 ? inv : nullptr;  // X0 is u itself: A = s^2 u u^T
        if (hm::launch_ns_gemm(x_map[cur], x_map[cur], g1, 128, 0, st) != cudaSuccess) return HM_ERR_CUDA;

        hm::GemmParams g2 = g1;
        g2.unit_scale = nullptr;
        g2.K = c.mp;
        g2.epi = hm::kEpiPoly; g2.alpha = hp->ns_c; g2.beta = hp->ns_b;
        g2.add = bf(c.a_off); g2.add_us = g1.out_us; g2.ld_add = c.mp;
        g2.out = bf(c.b_off);
        if (hm::launch_ns_gemm(a_map, a_map, g2, 128, 0, st) != cudaSuccess) return HM_ERR_CUDA;

        const bool last = it + 1 == hp->ns_steps;
        hm::GemmParams g3{};
        g3.M = c.mp; g3.N = c.np; g3.K = c.mp; g3.units = 1;
        g3.epi = last ? hm::kEpiFinal : hm::kEpiUpdate; g3.alpha = 1.f; g3.beta = hp->ns_a;
        g3.add = bf(c.x_off[cur]); g3.add_us = static_cast<int64_t>(c.mp) * c.np; g3.ld_add = c.np;
        g3.out = bf(c.x_off[cur ^ 1]); g3.out_us = g3.add_us; g3.ld_out = c.np;
        g3.ns_units = unit_dev; g3.v_root = v; g3.v_stage = nullptr;
        g3.m_real = m; g3.n_real = n;
        g3.err = g1.err;
        g3.unit_scale = it == 0 ? inv : nullptr;  // X1 = s (a u + B u)
        if (hm::launch_ns_gemm(b_map, x_mn[cur], g3, bn3, 1, st) != cudaSuccess) return HM_ERR_CUDA;
        cur ^= 1;
    }
    return HM_OK;
}
