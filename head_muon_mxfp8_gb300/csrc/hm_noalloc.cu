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
// muon_update_units for a unit whose smaller side is at most 128: the same
// prepare and norm kernels and the same one-launch tcgen05 Newton-Schulz
// kernel, on the built-in scratch instead of a caller workspace.
#include "hm.h"
#include "hm_internal.h"

#include <mutex>

namespace {

constexpr int kMaxM = HM_NOALLOC_MAX_MIN_DIM;   // padded Gram size of the scratch
constexpr int kMaxN = HM_NOALLOC_MAX_MAX_DIM;
constexpr size_t kSlot = 1024;
constexpr size_t kXBytes = static_cast<size_t>(kMaxM) * kMaxN * 2;
// one norm partial per 64 x 64 tile of X
constexpr size_t kPartsBytes = (static_cast<size_t>(kMaxM / 64) * (kMaxN / 64) * 4 + kSlot - 1) / kSlot * kSlot;
// layout: unit descriptor | X0 | X1 | partials | 1/norm  (A and B stay on chip)
constexpr size_t kOffUnit = 0;
constexpr size_t kOffX0 = kSlot;
constexpr size_t kOffX1 = kOffX0 + kXBytes;
constexpr size_t kOffParts = kOffX1 + kXBytes;
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
    c.part_off = kOffParts;
    c.inv_off = kOffInv;
    hm::NsUnit* unit_dev = reinterpret_cast<hm::NsUnit*>(ws + kOffUnit);

    CUtensorMap x_map[2];
    bool ok = true;
    for (int b = 0; b < 2; ++b) ok = ok && map_bf16(&x_map[b], ws + c.x_off[b], c.np, c.mp, 128);
    if (!ok) return HM_ERR_CUDA;

    hm::note_launch();
    write_unit_kernel<<<1, 1, 0, st>>>(unit_dev, unit);
    if (cudaGetLastError() != cudaSuccess) return HM_ERR_CUDA;
    if (hm::launch_ns_prepare(c, unit_dev, u, nullptr, ws, st) != cudaSuccess ||
        hm::launch_ns_norm(c, ws, hp->eps, st) != cudaSuccess)
        return HM_ERR_CUDA;
    // every product of every iteration in one kernel (the kernel
    // muon_update_units runs for Gram size 128), on the built-in X buffers
    hm::SmallNsParams sp{};
    sp.g.ns_units = unit_dev;
    sp.g.v_root = v;
    sp.g.m_real = m;
    sp.g.n_real = n;
    sp.g.err = hm::device_error_word();
    sp.g.unit_scale = reinterpret_cast<const float*>(ws + c.inv_off);
    sp.units = 1;
    sp.np = c.np;
    sp.steps = hp->ns_steps;
    sp.reverse = 1;
    sp.a = hp->ns_a;
    sp.b = hp->ns_b;
    sp.c = hp->ns_c;
    if (hm::launch_ns_small(x_map[0], x_map[1], sp, st) != cudaSuccess) return HM_ERR_CUDA;
    return HM_OK;
}
