// Host side of libhm: status codes, data tree, shard chain, Muon update
// planning, workspace layout, tensor-map encoding and stage orchestration.
//
// Follows "SS-HSDP: Efficient and Flexible Sharded Data Parallelism via
// Runtime-Update Decoupling": section 3.2 (Data Tree, Shard Chain,
// Distributed updates), section 3.4 (Execution Flow: the Update paragraph),
// section 4.1 (Batched Update and Transform), section 4.2 (Fully Zero Copy:
// hierarchical rank order of the ZeRO-1 shards) and Table 4 (planning rejects
// invalid geometry, incompatible metadata and storage overlap before any
// launch).
#include "hm.h"
#include "hm_internal.h"

#include <algorithm>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <new>
#include <utility>
#include <vector>

using hm::NsClassDev;
using hm::NsUnit;
using hm::NsFrag;
using hm::Range;
using hm::RangeArgs;

// ============================================================================
// status, device checks
// ============================================================================
extern "C" const char* hm_status_str(hm_status s) {
    switch (s) {
        case HM_OK: return "HM_OK";
        case HM_ERR_ARG: return "HM_ERR_ARG";
        case HM_ERR_GEOMETRY: return "HM_ERR_GEOMETRY";
        case HM_ERR_OVERLAP: return "HM_ERR_OVERLAP";
        case HM_ERR_ALIGN: return "HM_ERR_ALIGN";
        case HM_ERR_DTYPE: return "HM_ERR_DTYPE";
        case HM_ERR_UNITS: return "HM_ERR_UNITS";
        case HM_ERR_CUDA: return "HM_ERR_CUDA";
        case HM_ERR_ARCH: return "HM_ERR_ARCH";
        case HM_ERR_TIMEOUT: return "HM_ERR_TIMEOUT";
        case HM_ERR_WORKSPACE: return "HM_ERR_WORKSPACE";
        case HM_ERR_STATE: return "HM_ERR_STATE";
        default: return "HM_ERR_UNKNOWN";
    }
}

namespace {

// Unsupported hardware is rejected before any launch (Table 4).
hm_status check_arch() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return HM_ERR_CUDA;
    static std::mutex mu;
    static std::map<int, hm_status> cache;
    std::lock_guard<std::mutex> lk(mu);
    auto it = cache.find(dev);
    if (it != cache.end()) return it->second;
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return HM_ERR_CUDA;
    hm_status st = (major == 10 && minor == 3) ? HM_OK : HM_ERR_ARCH;
    cache[dev] = st;
    return st;
}

inline hm_status cuda_status(cudaError_t e) { return e == cudaSuccess ? HM_OK : HM_ERR_CUDA; }

size_t dtype_size(hm_dtype d) {
    switch (d) {
        case HM_U8: return 1;
        case HM_E4M3: return 1;
        case HM_BF16: return 2;
        case HM_F32: return 4;
        default: return 0;
    }
}

inline int64_t round_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" hm_status hm_kernel_launches(int64_t* count) {
    if (!count) return HM_ERR_ARG;
    *count = hm::launches_issued();
    return HM_OK;
}

extern "C" hm_status hm_device_error(int* code) {
    if (!code) return HM_ERR_ARG;
    hm_status st = check_arch();
    if (st != HM_OK) return st;
    int32_t* word = hm::device_error_word();
    if (!word) return HM_ERR_CUDA;
    int32_t v = 0, zero = 0;
    if (cudaDeviceSynchronize() != cudaSuccess) return HM_ERR_CUDA;
    if (cudaMemcpy(&v, word, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return HM_ERR_CUDA;
    if (cudaMemcpy(word, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return HM_ERR_CUDA;
    *code = v;
    return HM_OK;
}

// ============================================================================
// Data tree (section 3.2, "Data Tree")
// ============================================================================
struct hm_tree {
    struct Node {
        int parent;
        size_t acc;     // accumulated byte offset from the root
        size_t nbytes;
        hm_dtype dtype;
    };
    char* root;
    std::vector<Node> nodes;
};

extern "C" hm_status create_data_tree(hm_tree** out, void* root, size_t root_bytes) {
    if (!out || !root || root_bytes == 0) return HM_ERR_ARG;
    hm_tree* t = new (std::nothrow) hm_tree;
    if (!t) return HM_ERR_ARG;
    t->root = static_cast<char*>(root);
    t->nodes.push_back({-1, 0, root_bytes, HM_U8});
    *out = t;
    return HM_OK;
}

extern "C" hm_status data_tree_add_view(hm_tree* t, int parent, size_t byte_off, hm_dtype dtype,
                                        int ndim, const int64_t* shape, int* node_out) {
    if (!t || !shape || !node_out || ndim < 1 || ndim > 8) return HM_ERR_ARG;
    if (parent < 0 || parent >= static_cast<int>(t->nodes.size())) return HM_ERR_ARG;
    size_t es = dtype_size(dtype);
    if (es == 0) return HM_ERR_DTYPE;
    size_t numel = 1;
    for (int i = 0; i < ndim; ++i) {
        if (shape[i] < 0) return HM_ERR_ARG;
        if (shape[i] > 0 && numel > (SIZE_MAX / 16) / static_cast<size_t>(shape[i])) return HM_ERR_GEOMETRY;
        numel *= static_cast<size_t>(shape[i]);
    }
    const hm_tree::Node& p = t->nodes[parent];
    size_t nbytes = numel * es;
    if (byte_off > p.nbytes || nbytes > p.nbytes - byte_off) return HM_ERR_GEOMETRY;
    size_t acc = p.acc + byte_off;
    if (acc % es) return HM_ERR_ALIGN;
    t->nodes.push_back({parent, acc, nbytes, dtype});
    *node_out = static_cast<int>(t->nodes.size()) - 1;
    return HM_OK;
}

extern "C" hm_status data_tree_resolve(const hm_tree* t, int node, void** ptr, size_t* root_off) {
    if (!t || node < 0 || node >= static_cast<int>(t->nodes.size())) return HM_ERR_ARG;
    const size_t acc = t->nodes[node].acc;  // root + accumulated offset
    if (ptr) *ptr = t->root + acc;
    if (root_off) *root_off = acc;
    return HM_OK;
}

extern "C" hm_status data_tree_check_disjoint(const hm_tree* t, const int* nodes, int n) {
    if (!t || (n > 0 && !nodes) || n < 0) return HM_ERR_ARG;
    std::vector<std::pair<size_t, size_t>> iv;
    for (int i = 0; i < n; ++i) {
        if (nodes[i] < 0 || nodes[i] >= static_cast<int>(t->nodes.size())) return HM_ERR_ARG;
        const hm_tree::Node& x = t->nodes[nodes[i]];
        if (x.nbytes) iv.push_back({x.acc, x.acc + x.nbytes});
    }
    std::sort(iv.begin(), iv.end());
    for (size_t i = 1; i < iv.size(); ++i)
        if (iv[i].first < iv[i - 1].second) return HM_ERR_OVERLAP;
    return HM_OK;
}

extern "C" void tree_destroy(hm_tree* t) { delete t; }

// ============================================================================
// Shard chain (section 3.2 "Shard Chain"; section 4.2 rank order)
// ============================================================================
struct hm_chain {
    int64_t n = 0;
    int so = 1, sw = 1, sg = 1;
    std::vector<int64_t> edges;   // so + 1 z1 edges
    std::vector<int> owner;       // z1 chunk -> rank
    std::vector<int> chunk_of;    // rank -> z1 chunk
    std::vector<int64_t> base;    // rank -> segment element offset in the root
    std::vector<int64_t> len;     // rank -> segment length
    int64_t total = 0;            // elements of one emulated root
};

extern "C" hm_status shard_chain(hm_chain** out, int64_t n, int so, int sw, int sg,
                                 const int64_t* z1_edges, const int64_t* edge_shift) {
    if (!out || n < 0 || so < 1 || sw < 1 || sg < 1 || so > 4096) return HM_ERR_ARG;
    if (z1_edges && edge_shift) return HM_ERR_ARG;
    if (edge_shift) {
        if (edge_shift[0] != 0 || edge_shift[so] != 0) return HM_ERR_GEOMETRY;
        for (int i = 0; i <= so; ++i)
            if (edge_shift[i] % HM_MX_BLOCK) return HM_ERR_ALIGN;
    }
    if (n % HM_MX_BLOCK) return HM_ERR_ALIGN;
    if (sg % sw || so % sg) return HM_ERR_GEOMETRY;  // nested degrees (Table 4)
    hm_chain* c = new (std::nothrow) hm_chain;
    if (!c) return HM_ERR_ARG;
    c->n = n;
    c->so = so;
    c->sw = sw;
    c->sg = sg;
    c->edges.resize(so + 1);
    for (int i = 0; i <= so; ++i)
        c->edges[i] = z1_edges ? z1_edges[i]
                               : 32 * ((static_cast<int64_t>(i) * n) / (32LL * so)) + (edge_shift ? edge_shift[i] : 0);
    hm_status bad = HM_OK;
    if (c->edges[0] != 0 || c->edges[so] != n) bad = HM_ERR_GEOMETRY;
    for (int i = 0; i < so && bad == HM_OK; ++i) {
        if (c->edges[i + 1] < c->edges[i]) bad = HM_ERR_GEOMETRY;
        if (c->edges[i] % HM_MX_BLOCK) bad = HM_ERR_ALIGN;
    }
    if (bad != HM_OK) {
        delete c;
        return bad;
    }
    const int R = so / sw;
    c->owner.resize(so);
    c->chunk_of.resize(so);
    for (int ch = 0; ch < so; ++ch) {
        int r = ch / R + (ch % R) * sw;
        c->owner[ch] = r;
        c->chunk_of[r] = ch;
    }
    c->base.resize(so);
    c->len.resize(so);
    int64_t pos = HM_SEG_GAP;
    for (int r = 0; r < so; ++r) {
        int ch = c->chunk_of[r];
        c->base[r] = pos;
        c->len[r] = c->edges[ch + 1] - c->edges[ch];
        pos += round_up(c->len[r], HM_SEG_ALIGN) + HM_SEG_GAP;
    }
    c->total = pos;
    *out = c;
    return HM_OK;
}

extern "C" hm_status shard_chain_layout(const hm_chain* c, int64_t* total, int64_t* bases,
                                        int64_t* lens, int32_t* chunk_of_rank) {
    if (!c) return HM_ERR_ARG;
    if (total) *total = c->total;
    for (int r = 0; r < c->so; ++r) {
        if (bases) bases[r] = c->base[r];
        if (lens) lens[r] = c->len[r];
        if (chunk_of_rank) chunk_of_rank[r] = c->chunk_of[r];
    }
    return HM_OK;
}

namespace {

std::vector<hm_fragment> fragments_of(const hm_chain* c, int64_t a, int64_t b, int level) {
    std::vector<hm_fragment> out;
    const int s = level == 1 ? c->so : (level == 2 ? c->sg : c->sw);
    const int per = c->so / s;
    for (int k = 0; k < s; ++k) {
        const int64_t e0 = c->edges[k * per], e1 = c->edges[(k + 1) * per];
        const int64_t lo = std::max(a, e0), hi = std::min(b, e1);
        if (lo >= hi) continue;
        hm_fragment f;
        f.chunk = k;
        if (level == 1) {
            f.rank = c->owner[k];
            f.root_offset = c->base[f.rank] + (lo - e0);
        } else {
            int r = 0;
            while (c->chunk_of[r] / per != k) ++r;  // lowest rank holding chunk k
            f.rank = r;
            f.root_offset = -1;
        }
        f.seg_offset = lo - e0;
        f.unit_offset = lo - a;
        f.length = hi - lo;
        out.push_back(f);
    }
    return out;
}

}  // namespace

extern "C" hm_status shard_chain_fragments(const hm_chain* c, int64_t a, int64_t b, int level,
                                           hm_fragment* out, int cap, int* n) {
    if (!c || !n || level < 1 || level > 3 || cap < 0 || (cap > 0 && !out)) return HM_ERR_ARG;
    if (a < 0 || b < a || b > c->n) return HM_ERR_GEOMETRY;
    std::vector<hm_fragment> f = fragments_of(c, a, b, level);
    for (int i = 0; i < static_cast<int>(f.size()) && i < cap; ++i) out[i] = f[i];
    *n = static_cast<int>(f.size());
    return HM_OK;
}

extern "C" hm_status shard_chain_segment_views(const hm_chain* c, hm_tree* t, hm_dtype dtype,
                                               int* nodes_out) {
    if (!c || !t || !nodes_out) return HM_ERR_ARG;
    size_t es = dtype_size(dtype);
    if (!es) return HM_ERR_DTYPE;
    for (int r = 0; r < c->so; ++r) {
        int64_t shape = c->len[r];
        hm_status st = data_tree_add_view(t, 0, static_cast<size_t>(c->base[r]) * es, dtype, 1, &shape,
                                          &nodes_out[r]);
        if (st != HM_OK) return st;
    }
    return HM_OK;
}

extern "C" void chain_destroy(hm_chain* c) { delete c; }

// ============================================================================
// Muon plan (section 3.2 "Distributed updates"; section 3.4; section 4.1)
// ============================================================================
namespace {

constexpr size_t kWsAlign = 1024;

struct UnitPlan {
    int exec_rank = 0;
    int cls = 0;
    int local = 1;
    int64_t stage_off = -1;   // element offset in the u / v staging (straddling units)
    bool epi = false;         // the last Newton-Schulz product can apply f2 + G itself (kNsEpiUpdate)
    std::vector<hm_fragment> frags;
};

struct ClassMaps {
    CUtensorMap x_a[2], x_b[2], a_a, a_b, b_a, x_mn[2];
    int bn1 = 128, bn3 = 128;
};

double alpha_of(int mode, int rows, int cols) {
    if (mode == 1) return std::sqrt(std::max(1.0, static_cast<double>(rows) / cols));
    if (mode == 2) return 0.2 * std::sqrt(static_cast<double>(std::max(rows, cols)));
    return 1.0;
}

}  // namespace

struct hm_muon_plan {
    hm_chain chain;
    std::vector<std::vector<int32_t>> sym_tab;  // per class: triangular tile list
    std::vector<std::vector<int32_t>> pair_tab; // per class: the same for 256 x 256 tiles
    std::vector<hm_unit_desc> units;
    std::vector<UnitPlan> up;
    std::vector<NsClassDev> classes;
    std::vector<NsUnit> ns_units;
    std::vector<Range> seg_tab, gather_tab;
    mutable std::vector<Range> f2_tab;
    std::vector<std::pair<int, int>> f2_shape;  // (rows, cols) of each f2 entry's unit
    // HM_STAGE_SCRATCH: the f2 entries of units the last product cannot update
    // itself, and every unit's fragments for the ones it can
    mutable std::vector<Range> f2r_tab;
    std::vector<std::pair<int, int>> f2r_shape;
    mutable std::vector<NsUnit> ns_units_dev;  // ns_units with the current steps
    std::vector<NsFrag> ns_frags;
    size_t off_f2r = 0, off_nsf = 0;
    // fused update: f0 with the gather folded in (f2 + G reuse the f2 table)
    std::vector<Range> f0x_tab;
    size_t off_f0x = 0;
    int64_t staging_elems = 0;
    int n_straddling = 0, n_frag = 0;
    size_t off_seg = 0, off_gather = 0, off_f2 = 0, off_nsu = 0, off_ustage = 0, off_vstage = 0;
    size_t off_pace = 0;  // two ints pacing the CTA-pair GEMMs (zeroed at upload, kept zero between launches)
    size_t ws_bytes = 0;
    // upload state
    char* ws = nullptr;
    std::vector<ClassMaps> maps;
    mutable float f2_lr = NAN;
    // f0 ran with u as scratch: X0 and the unit scales of every class are in the
    // workspace, so the next Newton-Schulz stage skips the prepare pass
    mutable bool x0_ready = false;
    mutable int f2_alpha_mode = -1;
};

extern "C" hm_status muon_plan(hm_muon_plan** out, const hm_chain* chain, const hm_unit_desc* units,
                               int n_units) {
    if (!out || !chain || n_units < 0 || (n_units > 0 && !units)) return HM_ERR_ARG;
    // units must tile [0, n) in order (Appendix A: fields describe the same units)
    int64_t pos = 0;
    for (int i = 0; i < n_units; ++i) {
        const hm_unit_desc& u = units[i];
        if (u.rows < 1 || u.cols < 1 || u.rows > (1 << 20) || u.cols > (1 << 20)) return HM_ERR_GEOMETRY;
        if (u.offset != pos) return HM_ERR_UNITS;
        int64_t ne = static_cast<int64_t>(u.rows) * u.cols;
        if (ne % HM_MX_BLOCK) return HM_ERR_ALIGN;
        pos += ne;
    }
    if (pos != chain->n) return HM_ERR_UNITS;

    hm_muon_plan* p = new (std::nothrow) hm_muon_plan;
    if (!p) return HM_ERR_ARG;
    p->chain = *chain;
    p->units.assign(units, units + n_units);
    p->up.resize(n_units);

    std::map<std::pair<int, int>, int> cls_of;
    std::vector<std::vector<int>> members;
    for (int i = 0; i < n_units; ++i) {
        const hm_unit_desc& u = units[i];
        UnitPlan& q = p->up[i];
        int64_t ne = static_cast<int64_t>(u.rows) * u.cols;
        q.frags = fragments_of(chain, u.offset, u.offset + ne, 1);
        q.local = q.frags.size() == 1;
        q.exec_rank = q.frags[0].rank;  // owner of the unit's first element
        // each 1 x 32 MX block a row piece inside one fragment
        q.epi = u.cols % HM_MX_BLOCK == 0;
        for (const hm_fragment& f : q.frags)
            q.epi = q.epi && f.root_offset % HM_MX_BLOCK == 0 && f.unit_offset % HM_MX_BLOCK == 0 &&
                    f.length % HM_MX_BLOCK == 0;
        if (!q.local) {
            q.stage_off = p->staging_elems;
            p->staging_elems += round_up(ne, 64);
            p->n_straddling++;
            p->n_frag += static_cast<int>(q.frags.size());
        }
        std::pair<int, int> key(std::min(u.rows, u.cols), std::max(u.rows, u.cols));
        auto it = cls_of.find(key);
        if (it == cls_of.end()) {
            it = cls_of.emplace(key, static_cast<int>(members.size())).first;
            members.emplace_back();
        }
        q.cls = it->second;
        members[q.cls].push_back(i);
    }

    // Newton-Schulz unit table, grouped by shape class (section 4.1: matrices
    // with matching shapes are grouped for batched GEMMs)
    for (size_t k = 0; k < members.size(); ++k) {
        if (members[k].size() > 65535) {  // a class's units span one grid dimension
            delete p;
            return HM_ERR_GEOMETRY;
        }
        NsClassDev c{};
        const hm_unit_desc& u0 = units[members[k][0]];
        c.m = std::min(u0.rows, u0.cols);
        c.n = std::max(u0.rows, u0.cols);
        c.mp = static_cast<int32_t>(round_up(c.m, 128));
        c.np = static_cast<int32_t>(round_up(c.n, 64));
        c.n_units = static_cast<int32_t>(members[k].size());
        c.first_unit = static_cast<int32_t>(p->ns_units.size());
        // A = X X^T and B = bA + cAA are symmetric: only output tiles with an
        // element on or above the diagonal are computed (the epilogue mirrors
        // them).  Order: bands of 8 tile-rows, column by column in a band.
        {
            const int bn = c.mp >= 256 ? 256 : 128;
            const int tiles_m = c.mp / 128, tiles_n = (c.mp + bn - 1) / bn;
            std::vector<int32_t> tab;
            for (int g0 = 0; g0 < tiles_m; g0 += 8)
                for (int tn = 0; tn < tiles_n; ++tn)
                    for (int tm = g0; tm < std::min(tiles_m, g0 + 8); ++tm)
                        if (tn * bn + bn - 1 >= tm * 128) tab.push_back((tm << 16) | tn);
            c.sym_tiles = static_cast<int32_t>(tab.size());
            p->sym_tab.push_back(tab);
            // 256 x 256 tiles (CTA pairs): tn >= tm, bands of 4 tile-rows
            std::vector<int32_t> tab2;
            const int t2 = (c.mp + 255) / 256;
            for (int g0 = 0; g0 < t2; g0 += 4)
                for (int tn = 0; tn < t2; ++tn)
                    for (int tm = g0; tm < std::min(t2, g0 + 4); ++tm)
                        if (tn >= tm) tab2.push_back((tm << 16) | tn);
            c.pair_tiles = static_cast<int32_t>(tab2.size());
            p->pair_tab.push_back(tab2);
        }
        c.parts = (c.np / 64) * (c.mp / 64);  // one sum of squares per 64 x 64 tile of X
        for (int i : members[k]) {
            const hm_unit_desc& u = units[i];
            const UnitPlan& q = p->up[i];
            NsUnit nu{};
            nu.rows = u.rows;
            nu.cols = u.cols;
            nu.u_off = q.local ? q.frags[0].root_offset : q.stage_off;
            nu.v_off = nu.u_off;
            nu.flags = (q.local ? 0 : (hm::kNsUStaged | hm::kNsVStaged)) |
                       (u.rows > u.cols ? hm::kNsTransposed : 0);
            if (q.epi) nu.flags |= hm::kNsEpiUpdate;
            // every unit's fragments: f0 folded into the prepare pass reads g and m
            // through them; the last product's f2 + G writes w, q and s through them
            nu.frag0 = static_cast<int32_t>(p->ns_frags.size());
            nu.nfrag = static_cast<int32_t>(q.frags.size());
            for (const hm_fragment& f : q.frags) p->ns_frags.push_back(NsFrag{f.unit_offset, f.root_offset});
            p->ns_units.push_back(nu);
        }
        p->classes.push_back(c);
    }

    // range tables
    int64_t pre = 0;
    for (int r = 0; r < chain->so; ++r) {
        if (!chain->len[r]) continue;
        Range g{chain->base[r], chain->base[r], chain->base[r], chain->len[r], pre, 0.f, 0};
        p->seg_tab.push_back(g);
        pre += chain->len[r];
    }
    pre = 0;
    for (int i = 0; i < n_units; ++i) {
        const UnitPlan& q = p->up[i];
        if (q.local) continue;
        for (const hm_fragment& f : q.frags) {
            p->gather_tab.push_back(Range{f.root_offset, q.stage_off + f.unit_offset, 0, f.length, pre, 0.f, 0});
            pre += f.length;
        }
    }
    pre = 0;
    for (int i = 0; i < n_units; ++i) {
        const hm_unit_desc& u = units[i];
        const UnitPlan& q = p->up[i];
        if (q.local) {
            const hm_fragment& f = q.frags[0];
            if (!p->f2_tab.empty()) {
                Range& last = p->f2_tab.back();
                if (last.flags == 0 && last.a + last.len == f.root_offset &&
                    p->f2_shape.back() == std::make_pair(u.rows, u.cols)) {
                    last.len += f.length;
                    pre += f.length;
                    continue;
                }
            }
            p->f2_tab.push_back(Range{f.root_offset, f.root_offset, f.root_offset, f.length, pre, 0.f, 0});
            p->f2_shape.push_back({u.rows, u.cols});
            pre += f.length;
        } else {
            for (const hm_fragment& f : q.frags) {
                p->f2_tab.push_back(Range{f.root_offset, q.stage_off + f.unit_offset, f.root_offset, f.length, pre,
                                          0.f, 1});
                p->f2_shape.push_back({u.rows, u.cols});
                pre += f.length;
            }
        }
    }
    pre = 0;
    for (int i = 0; i < n_units; ++i) {
        const hm_unit_desc& u = units[i];
        const UnitPlan& q = p->up[i];
        if (q.epi) continue;
        for (const hm_fragment& f : q.frags) {
            p->f2r_tab.push_back(Range{f.root_offset, q.local ? f.root_offset : q.stage_off + f.unit_offset,
                                       f.root_offset, f.length, pre, 0.f, q.local ? 0 : 1});
            p->f2r_shape.push_back({u.rows, u.cols});
            pre += f.length;
        }
    }

    // fused-update tables
    pre = 0;
    for (int i = 0; i < n_units; ++i) {
        const UnitPlan& q = p->up[i];
        for (const hm_fragment& f : q.frags) {
            if (q.local && !p->f0x_tab.empty()) {
                Range& last = p->f0x_tab.back();
                if (last.flags == 0 && last.a + last.len == f.root_offset) {
                    last.len += f.length;
                    pre += f.length;
                    continue;
                }
            }
            p->f0x_tab.push_back(Range{f.root_offset, q.local ? 0 : q.stage_off + f.unit_offset, 0, f.length, pre,
                                       0.f, q.local ? 0 : 2});
            pre += f.length;
        }
    }

    // workspace layout (every region 1024-byte aligned)
    size_t off = 0;
    auto take = [&](size_t bytes) {
        size_t at = off;
        off += (bytes + kWsAlign - 1) / kWsAlign * kWsAlign;
        return at;
    };
    p->off_seg = take(p->seg_tab.size() * sizeof(Range));
    p->off_gather = take(p->gather_tab.size() * sizeof(Range));
    p->off_f2 = take(p->f2_tab.size() * sizeof(Range));
    p->off_nsu = take(p->ns_units.size() * sizeof(NsUnit));
    p->off_f2r = take(p->f2r_tab.size() * sizeof(Range));
    p->off_nsf = take(p->ns_frags.size() * sizeof(NsFrag));
    p->off_f0x = take(p->f0x_tab.size() * sizeof(Range));
    p->off_ustage = take(static_cast<size_t>(p->staging_elems) * 2);
    p->off_vstage = take(static_cast<size_t>(p->staging_elems) * 4);
    p->off_pace = take(2 * sizeof(int32_t));
    for (NsClassDev& c : p->classes) {
        size_t xb = static_cast<size_t>(c.n_units) * c.mp * c.np * 2;
        size_t ab = static_cast<size_t>(c.n_units) * c.mp * c.mp * 2;
        c.x_off[0] = take(xb);
        c.x_off[1] = take(xb);
        c.a_off = take(ab);
        c.b_off = take(ab);
        c.part_off = take(static_cast<size_t>(c.n_units) * c.parts * 4);
        c.inv_off = take(static_cast<size_t>(c.n_units) * 4);
        c.sym_off = take(static_cast<size_t>(c.sym_tiles) * 4);
        c.pair_off = take(static_cast<size_t>(c.pair_tiles) * 4);
    }
    p->ws_bytes = std::max<size_t>(off, kWsAlign);
    *out = p;
    return HM_OK;
}

extern "C" hm_status muon_plan_query(const hm_muon_plan* p, hm_muon_plan_info* info) {
    if (!p || !info) return HM_ERR_ARG;
    info->n_units = static_cast<int32_t>(p->units.size());
    info->n_straddling = p->n_straddling;
    info->n_local = info->n_units - p->n_straddling;
    info->n_classes = static_cast<int32_t>(p->classes.size());
    info->staging_elems = p->staging_elems;
    info->workspace_bytes = static_cast<int64_t>(p->ws_bytes);
    info->n_fragments = p->n_frag;
    return HM_OK;
}

extern "C" hm_status muon_plan_unit(const hm_muon_plan* p, int unit, int32_t* exec_rank, int32_t* n_frags,
                                    int32_t* cls, int32_t* local) {
    if (!p || unit < 0 || unit >= static_cast<int>(p->units.size())) return HM_ERR_ARG;
    const UnitPlan& q = p->up[unit];
    if (exec_rank) *exec_rank = q.exec_rank;
    if (n_frags) *n_frags = static_cast<int32_t>(q.frags.size());
    if (cls) *cls = q.cls;
    if (local) *local = q.local;
    return HM_OK;
}

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                   CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(f);
    });
    return fn;
}

// 3-D bf16 tensor [units][rows][inner] (inner contiguous), tile box
// [1][box_rows][64] with the 128-byte swizzle the UMMA K-major layout expects.
bool encode_bf16_3d(CUtensorMap* m, void* base, int64_t inner, int64_t rows, int64_t units, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows),
                          static_cast<cuuint64_t>(units)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(inner * 2), static_cast<cuuint64_t>(inner * rows * 2)};
    cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_rows), 1};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

RangeArgs device_ranges(const char* ws, size_t off, const std::vector<Range>& tab) {
    RangeArgs ra;
    std::memset(&ra, 0, sizeof(ra));
    ra.tab = reinterpret_cast<const Range*>(ws + off);
    ra.n = static_cast<int32_t>(tab.size());
    ra.total = tab.empty() ? 0 : tab.back().prefix + tab.back().len;
    return ra;
}

}  // namespace

extern "C" hm_status muon_plan_upload(hm_muon_plan* p, void* workspace, size_t workspace_bytes, void* stream) {
    if (!p || !workspace) return HM_ERR_ARG;
    hm_status st = check_arch();
    if (st != HM_OK) return st;
    if (workspace_bytes < p->ws_bytes || (reinterpret_cast<uintptr_t>(workspace) % kWsAlign))
        return HM_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    char* ws = static_cast<char*>(workspace);
    auto put = [&](size_t off, const void* src, size_t bytes) {
        return bytes == 0 ? cudaSuccess : cudaMemcpyAsync(ws + off, src, bytes, cudaMemcpyHostToDevice, s);
    };
    if (put(p->off_seg, p->seg_tab.data(), p->seg_tab.size() * sizeof(Range)) != cudaSuccess ||
        put(p->off_gather, p->gather_tab.data(), p->gather_tab.size() * sizeof(Range)) != cudaSuccess ||
        put(p->off_nsu, p->ns_units.data(), p->ns_units.size() * sizeof(NsUnit)) != cudaSuccess ||
        put(p->off_nsf, p->ns_frags.data(), p->ns_frags.size() * sizeof(NsFrag)) != cudaSuccess)
        return HM_ERR_CUDA;
    for (size_t k = 0; k < p->classes.size(); ++k)
        if (put(p->classes[k].sym_off, p->sym_tab[k].data(), p->sym_tab[k].size() * 4) != cudaSuccess ||
            put(p->classes[k].pair_off, p->pair_tab[k].data(), p->pair_tab[k].size() * 4) != cudaSuccess)
            return HM_ERR_CUDA;
    if (put(p->off_f0x, p->f0x_tab.data(), p->f0x_tab.size() * sizeof(Range)) != cudaSuccess) return HM_ERR_CUDA;
    if (cudaMemsetAsync(ws + p->off_pace, 0, 2 * sizeof(int32_t), s) != cudaSuccess) return HM_ERR_CUDA;
    p->maps.assign(p->classes.size(), ClassMaps{});
    for (size_t k = 0; k < p->classes.size(); ++k) {
        const NsClassDev& c = p->classes[k];
        ClassMaps& mp = p->maps[k];
        mp.bn1 = c.mp >= 256 ? 256 : 128;
        mp.bn3 = c.np >= 256 ? 256 : 128;
        bool ok = true;
        for (int b = 0; b < 2; ++b) {
            ok = ok && encode_bf16_3d(&mp.x_a[b], ws + c.x_off[b], c.np, c.mp, c.n_units, 128);
            ok = ok && encode_bf16_3d(&mp.x_b[b], ws + c.x_off[b], c.np, c.mp, c.n_units, mp.bn1);
            ok = ok && encode_bf16_3d(&mp.x_mn[b], ws + c.x_off[b], c.np, c.mp, c.n_units, 64);
        }
        ok = ok && encode_bf16_3d(&mp.a_a, ws + c.a_off, c.mp, c.mp, c.n_units, 128);
        ok = ok && encode_bf16_3d(&mp.a_b, ws + c.a_off, c.mp, c.mp, c.n_units, mp.bn1);
        ok = ok && encode_bf16_3d(&mp.b_a, ws + c.b_off, c.mp, c.mp, c.n_units, 128);
        if (!ok) return HM_ERR_CUDA;
    }
    p->ws = ws;
    p->f2_lr = NAN;  // force the f2 steps to be written on the next update
    p->x0_ready = false;
    p->f2_alpha_mode = -1;
    return HM_OK;
}

extern "C" hm_status muon_plan_staging(const hm_muon_plan* p, int unit, uint16_t** u_stage, float** v_stage) {
    if (!p || unit < 0 || unit >= static_cast<int>(p->units.size())) return HM_ERR_ARG;
    if (!p->ws) return HM_ERR_STATE;
    const UnitPlan& q = p->up[unit];
    if (q.local) return HM_ERR_ARG;
    if (u_stage) *u_stage = reinterpret_cast<uint16_t*>(p->ws + p->off_ustage) + q.stage_off;
    if (v_stage) *v_stage = reinterpret_cast<float*>(p->ws + p->off_vstage) + q.stage_off;
    return HM_OK;
}

namespace {

// Per-unit steps fp32(lr * alpha) live in the f2 table; it is rewritten (and
// re-uploaded, stream-ordered) whenever lr or the alpha mode changes.
hm_status refresh_steps(const hm_muon_plan* p, const hm_muon_hparams* hp, cudaStream_t s) {
    if (hp->lr == p->f2_lr && hp->alpha_mode == p->f2_alpha_mode) return HM_OK;
    auto step_of = [&](int rows, int cols) {
        return static_cast<float>(static_cast<double>(hp->lr) * alpha_of(hp->alpha_mode, rows, cols));
    };
    for (size_t i = 0; i < p->f2_tab.size(); ++i) p->f2_tab[i].step = step_of(p->f2_shape[i].first, p->f2_shape[i].second);
    for (size_t i = 0; i < p->f2r_tab.size(); ++i)
        p->f2r_tab[i].step = step_of(p->f2r_shape[i].first, p->f2r_shape[i].second);
    p->ns_units_dev = p->ns_units;
    for (NsUnit& nu : p->ns_units_dev) nu.step = step_of(nu.rows, nu.cols);
    auto put = [&](size_t off, const void* src, size_t bytes) {
        return bytes == 0 || cudaMemcpyAsync(p->ws + off, src, bytes, cudaMemcpyHostToDevice, s) == cudaSuccess;
    };
    if (!put(p->off_f2, p->f2_tab.data(), p->f2_tab.size() * sizeof(Range)) ||
        !put(p->off_f2r, p->f2r_tab.data(), p->f2r_tab.size() * sizeof(Range)) ||
        !put(p->off_nsu, p->ns_units_dev.data(), p->ns_units_dev.size() * sizeof(NsUnit)))
        return HM_ERR_CUDA;
    p->f2_lr = hp->lr;
    p->f2_alpha_mode = hp->alpha_mode;
    return HM_OK;
}

}  // namespace

// L2 size of the current device (cached per device).
static int64_t device_l2_bytes() {
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 128 << 20;
    if (!cached[dev]) {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrL2CacheSize, dev) != cudaSuccess || v <= 0) v = 128 << 20;
        cached[dev] = v;
    }
    return cached[dev];
}

extern "C" hm_status muon_update_units(const hm_muon_plan* p, const hm_muon_bufs* b, const hm_muon_hparams* hp,
                                       void* workspace, size_t workspace_bytes, int stages, void* stream) {
    if (!p || !b || !hp || stages < 0 || stages > HM_STAGE_STEP) return HM_ERR_ARG;
    const bool fused = stages & HM_STAGE_FUSED;
    // u and v as scratch: the fused passes only, and v may stay unwritten only
    // when the same call runs every stage that reads it
    const bool skip_v = stages & HM_STAGE_SCRATCH;
    const int v_needs = HM_STAGE_NS | HM_STAGE_F2 | HM_STAGE_REQUANT;
    if (skip_v && (!fused || ((stages & HM_STAGE_NS) && (stages & v_needs) != v_needs))) return HM_ERR_ARG;
    // the last products update the kNsEpiUpdate units themselves only when this
    // call also runs f2 + G for the rest
    const bool epi_update = skip_v && (stages & HM_STAGE_NS);
    if (fused) {
        // the fused passes cross stage boundaries: f0 + gather, and f2 + G
        const int front = stages & (HM_STAGE_F0 | HM_STAGE_GATHER);
        const int back = stages & (HM_STAGE_F2 | HM_STAGE_REQUANT);
        if ((front && front != (HM_STAGE_F0 | HM_STAGE_GATHER)) ||
            (back && back != (HM_STAGE_F2 | HM_STAGE_REQUANT)))
            return HM_ERR_ARG;
    }
    if (!p->ws) return HM_ERR_STATE;
    if (workspace != p->ws || workspace_bytes < p->ws_bytes) return HM_ERR_WORKSPACE;
    hm_status st = check_arch();
    if (st != HM_OK) return st;
    if ((stages & HM_STAGE_F0) && (!b->m || !b->g || !b->u)) return HM_ERR_ARG;
    if ((stages & HM_STAGE_GATHER) && !b->u) return HM_ERR_ARG;
    if ((stages & HM_STAGE_NS) && (!b->u || !b->v || hp->ns_steps < 1 || hp->ns_steps > 100)) return HM_ERR_ARG;
    if ((stages & HM_STAGE_F2) && (!b->w || !b->v || hp->alpha_mode < 0 || hp->alpha_mode > 2)) return HM_ERR_ARG;
    if ((stages & HM_STAGE_REQUANT) && (!b->w || !b->q || !b->s)) return HM_ERR_ARG;
    const void* ptrs[] = {b->w, b->m, b->g, b->u, b->v, b->q, b->s};
    for (const void* q : ptrs)
        if (q && !aligned16(q)) return HM_ERR_ALIGN;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    char* ws = p->ws;
    uint16_t* u_stage = reinterpret_cast<uint16_t*>(ws + p->off_ustage);
    float* v_stage = reinterpret_cast<float*>(ws + p->off_vstage);

    if ((stages & HM_STAGE_F2) && (st = refresh_steps(p, hp, s)) != HM_OK) return st;
    if (fused && (stages & HM_STAGE_F0) && skip_v) {
        // u as scratch: f0 runs inside the prepare pass of every shape class,
        // reading g and m through the units' fragments and writing X0 and the
        // norm's partial sums instead of u; the unit scales follow, and the next
        // Newton-Schulz stage on this plan starts from them
        const NsFrag* frags = reinterpret_cast<const NsFrag*>(ws + p->off_nsf);
        for (size_t k = 0; k < p->classes.size(); ++k) {
            const NsClassDev& c = p->classes[k];
            const NsUnit* units_dev = reinterpret_cast<const NsUnit*>(ws + p->off_nsu) + c.first_unit;
            if (hm::launch_ns_f0_prepare(c, units_dev, frags, b->m, b->g, hp->momentum, hp->nesterov, ws, s) !=
                    cudaSuccess ||
                hm::launch_ns_norm(c, ws, hp->eps, s) != cudaSuccess)
                return HM_ERR_CUDA;
        }
        p->x0_ready = true;
    } else if (fused && (stages & HM_STAGE_F0)) {
        // f0 writes u of straddling fragments into their staging as well
        RangeArgs ra = device_ranges(ws, p->off_f0x, p->f0x_tab);
        if (hm::launch_f0(ra, b->m, b->g, b->u, u_stage, hp->momentum, hp->nesterov, 0, s) != cudaSuccess)
            return HM_ERR_CUDA;
    }
    if ((stages & HM_STAGE_F0) && !(fused && skip_v)) p->x0_ready = false;  // u written: prepare from it
    if (!fused && (stages & HM_STAGE_F0)) {
        RangeArgs ra = device_ranges(ws, p->off_seg, p->seg_tab);
        if (hm::launch_f0(ra, b->m, b->g, b->u, nullptr, hp->momentum, hp->nesterov, 0, s) != cudaSuccess)
            return HM_ERR_CUDA;
    }
    if (!fused && (stages & HM_STAGE_GATHER) && !p->gather_tab.empty()) {
        RangeArgs ra = device_ranges(ws, p->off_gather, p->gather_tab);
        if (hm::launch_copy_bf16(ra, b->u, u_stage, s) != cudaSuccess) return HM_ERR_CUDA;
    }
    if (stages & HM_STAGE_NS) {
        // Failure-detection test hook: with HM_INJECT_NS_WAIT_TIMEOUT=1 in the
        // environment, the first GEMM of this call never marks an accumulator
        // ready, so its epilogue waits run out (bounded) and the kernel records
        // HM_ERR_TIMEOUT in the device error word.
        const char* inj = std::getenv("HM_INJECT_NS_WAIT_TIMEOUT");
        bool inject = inj && inj[0] == '1';
        const bool have_x0 = p->x0_ready;  // X0 and the unit scales left by f0 with u as scratch
        p->x0_ready = false;

        for (size_t k = 0; k < p->classes.size(); ++k) {
            const NsClassDev& c = p->classes[k];
            const ClassMaps& mp = p->maps[k];
            const NsUnit* units_dev = reinterpret_cast<const NsUnit*>(ws + p->off_nsu) + c.first_unit;
            if (!have_x0 && (hm::launch_ns_prepare(c, units_dev, b->u, u_stage, ws, s) != cudaSuccess ||
                             hm::launch_ns_norm(c, ws, hp->eps, s) != cudaSuccess))
                return HM_ERR_CUDA;
            const float* inv = reinterpret_cast<const float*>(ws + c.inv_off);
            if (c.mp == 128) {
                // Gram size 128 (the per-head units): every product of every
                // iteration in one persistent kernel, X read once and written once
                // per iteration, A and B kept on chip
                hm::SmallNsParams sp{};
                hm::GemmParams& g = sp.g;
                g.ns_units = units_dev; g.v_root = b->v; g.v_stage = v_stage;
                g.m_real = c.m; g.n_real = c.n;
                g.err = hm::device_error_word();
                g.inject_no_ready = inject ? 1 : 0;
                inject = false;
                g.unit_scale = inv;
                if (epi_update) {
                    g.fuse_update = 1;
                    g.decay = static_cast<float>(1.0 - static_cast<double>(hp->lr) * hp->weight_decay);
                    g.has_decay = hp->weight_decay != 0.f;
                    g.frags = reinterpret_cast<const NsFrag*>(ws + p->off_nsf);
                    g.w = b->w;
                    g.q = b->q;
                    g.s = b->s;
                }
                sp.units = c.n_units;
                sp.np = c.np;
                sp.steps = hp->ns_steps;
                sp.reverse = 1;
                sp.a = hp->ns_a;
                sp.b = hp->ns_b;
                sp.c = hp->ns_c;
                if (hm::launch_ns_small(mp.x_a[0], mp.x_a[1], sp, s) != cudaSuccess) return HM_ERR_CUDA;
                continue;
            }
            auto bf = [&](size_t off) { return reinterpret_cast<uint16_t*>(ws + off); };
            int cur = 0;
            for (int it = 0; it < hp->ns_steps; ++it) {
                hm::GemmParams g1{};
                g1.M = c.mp; g1.N = c.mp; g1.K = c.np; g1.units = c.n_units;
                g1.epi = hm::kEpiGram; g1.alpha = 1.f; g1.beta = 0.f;
                g1.out = bf(c.a_off); g1.out_us = static_cast<int64_t>(c.mp) * c.mp; g1.ld_out = c.mp;
                g1.err = hm::device_error_word();
                // pair pacing where it pays: units whose X is larger than half the
                // L2 (operand panels that drifting pairs would fetch from DRAM again);
                // small units stay cached anyway and only lose time to the waits
                const bool big_x = 2 * static_cast<int64_t>(c.mp) * c.np * 2 > device_l2_bytes();
                g1.pace = big_x ? reinterpret_cast<int32_t*>(ws + p->off_pace) : nullptr;
                g1.tile_tab = reinterpret_cast<const int32_t*>(ws + c.sym_off);
                g1.tab_len = c.sym_tiles;
                g1.sym = 1;
                g1.inject_no_ready = inject ? 1 : 0;
                g1.unit_scale = it == 0 ? inv : nullptr;  // X0 is u itself: A = s^2 u u^T
                inject = false;
                // classes whose Gram size is a multiple of 256 run on CTA pairs (256 x 256
                // tiles); others keep 128-row tiles, since a pair's last tile-row would be
                // half empty (1408-row experts: 1.5 % faster per update on single CTAs)
                const bool pair = c.mp >= 256 && c.mp % 256 == 0;
                if (pair) {
                    g1.tile_tab = reinterpret_cast<const int32_t*>(ws + c.pair_off);
                    g1.tab_len = c.pair_tiles;
                    if (hm::launch_ns_gemm_pair(mp.x_a[cur], mp.x_a[cur], g1, 0, s) != cudaSuccess) return HM_ERR_CUDA;
                } else if (hm::launch_ns_gemm(mp.x_a[cur], mp.x_b[cur], g1, mp.bn1, 0, s) != cudaSuccess) {
                    return HM_ERR_CUDA;
                }
                g1.inject_no_ready = 0;

                hm::GemmParams g2 = g1;
                g2.unit_scale = nullptr;
                g2.K = c.mp;
                g2.epi = hm::kEpiPoly; g2.alpha = hp->ns_c; g2.beta = hp->ns_b;
                g2.add = bf(c.a_off); g2.add_us = g1.out_us; g2.ld_add = c.mp;
                g2.out = bf(c.b_off);
                if (pair ? hm::launch_ns_gemm_pair(mp.a_a, mp.a_a, g2, 0, s) != cudaSuccess
                         : hm::launch_ns_gemm(mp.a_a, mp.a_b, g2, mp.bn1, 0, s) != cudaSuccess)
                    return HM_ERR_CUDA;

                const bool last = it + 1 == hp->ns_steps;
                hm::GemmParams g3{};
                g3.M = c.mp; g3.N = c.np; g3.K = c.mp; g3.units = c.n_units;
                g3.epi = last ? hm::kEpiFinal : hm::kEpiUpdate; g3.alpha = 1.f; g3.beta = hp->ns_a;
                g3.add = bf(c.x_off[cur]); g3.add_us = static_cast<int64_t>(c.mp) * c.np; g3.ld_add = c.np;
                g3.out = bf(c.x_off[cur ^ 1]); g3.out_us = g3.add_us; g3.ld_out = c.np;
                g3.ns_units = units_dev; g3.v_root = b->v; g3.v_stage = v_stage;
                g3.m_real = c.m; g3.n_real = c.n;
                g3.group_m = c.mp / 128;  // column bands: each X panel is fetched once per unit
                g3.err = g1.err;
                g3.pace = g1.pace;
                g3.unit_scale = it == 0 ? inv : nullptr;  // X1 = s (a u + B u)
                if (last && epi_update) {
                    // f2 and G of the kNsEpiUpdate units in this product's epilogue
                    g3.fuse_update = 1;
                    g3.decay = static_cast<float>(1.0 - static_cast<double>(hp->lr) * hp->weight_decay);
                    g3.has_decay = hp->weight_decay != 0.f;
                    g3.frags = reinterpret_cast<const NsFrag*>(ws + p->off_nsf);
                    g3.w = b->w;
                    g3.q = b->q;
                    g3.s = b->s;
                }
                if (pair) {
                    // B X raster for pairs: tile columns within bands of tile-rows, the
                    // fewest equal bands whose slab of B fits in a quarter of the L2 --
                    // that slab is re-read by every wave of its band and has to stay
                    // resident (5120 x 20480 class: two bands, 10.3 GB read per launch
                    // instead of 15.8 GB with one)
                    const int tiles_m = (c.mp + 255) / 256;
                    const int64_t b_bytes = static_cast<int64_t>(c.mp) * c.mp * 2;
                    const int64_t cap = std::max<int64_t>(device_l2_bytes() / 4, 1);
                    const int bands = static_cast<int>(std::min<int64_t>((b_bytes + cap - 1) / cap, tiles_m));
                    g3.group_m = (tiles_m + bands - 1) / bands;
                    if (hm::launch_ns_gemm_pair(mp.b_a, mp.x_mn[cur], g3, 1, s) != cudaSuccess) return HM_ERR_CUDA;
                } else if (hm::launch_ns_gemm(mp.b_a, mp.x_mn[cur], g3, mp.bn3, 1, s) != cudaSuccess) {
                    return HM_ERR_CUDA;
                }
                cur ^= 1;
            }
        }
    }
    if (fused && (stages & HM_STAGE_F2)) {
        // f2 and G in one pass: the new w of every element is quantized as it is
        // written (with HM_STAGE_SCRATCH only for units the last product left)
        const std::vector<Range>& tab = epi_update ? p->f2r_tab : p->f2_tab;
        if (!tab.empty()) {
            RangeArgs ra = device_ranges(ws, epi_update ? p->off_f2r : p->off_f2, tab);
            const float decay = static_cast<float>(1.0 - static_cast<double>(hp->lr) * hp->weight_decay);
            if (hm::launch_f2_requant(ra, b->w, b->v, v_stage, b->q, b->s, decay, hp->weight_decay != 0.f, s) !=
                cudaSuccess)
                return HM_ERR_CUDA;
        }
        return HM_OK;
    }
    if (stages & HM_STAGE_F2) {
        RangeArgs ra = device_ranges(ws, p->off_f2, p->f2_tab);
        const float decay = static_cast<float>(1.0 - static_cast<double>(hp->lr) * hp->weight_decay);
        if (hm::launch_f2(ra, b->w, b->v, v_stage, decay, hp->weight_decay != 0.f, s) != cudaSuccess)
            return HM_ERR_CUDA;
    }
    if (stages & HM_STAGE_REQUANT) {
        RangeArgs ra = device_ranges(ws, p->off_seg, p->seg_tab);
        if (hm::launch_requant(ra, b->w, b->q, b->s, s) != cudaSuccess) return HM_ERR_CUDA;
    }
    return HM_OK;
}

extern "C" void muon_plan_destroy(hm_muon_plan* p) { delete p; }

// ============================================================================
// AdamW (section 5.2) and MXFP8 requant (EG1)
// ============================================================================
extern "C" hm_status adamw_update_flat(float* w, const void* g, hm_dtype g_dtype, float* m, float* v, int64_t n,
                                       const hm_adamw_hparams* hp, void* stream) {
    if (n < 0 || !hp) return HM_ERR_ARG;
    if (g_dtype != HM_BF16 && g_dtype != HM_F32) return HM_ERR_DTYPE;
    if (hp->step < 1) return HM_ERR_ARG;
    if (n == 0) return HM_OK;
    if (!w || !g || !m || !v) return HM_ERR_ARG;
    if (!aligned16(w) || !aligned16(g) || !aligned16(m) || !aligned16(v)) return HM_ERR_ALIGN;
    hm_status st = check_arch();
    if (st != HM_OK) return st;
    const double bc1 = 1.0 - std::pow(static_cast<double>(hp->beta1), hp->step);
    const double bc2 = 1.0 - std::pow(static_cast<double>(hp->beta2), hp->step);
    const float decay = static_cast<float>(1.0 - static_cast<double>(hp->lr) * hp->weight_decay);
    const float step_size = static_cast<float>(hp->lr / bc1);
    const float inv_sqrt_bc2 = static_cast<float>(1.0 / std::sqrt(bc2));
    return cuda_status(hm::launch_adamw(w, g, g_dtype == HM_BF16, m, v, n, hp->lr, hp->beta1, hp->beta2, hp->eps,
                                        decay, step_size, inv_sqrt_bc2, static_cast<cudaStream_t>(stream)));
}

extern "C" hm_status mxfp8_requant_packed(const float* w, uint8_t* q, uint8_t* scales, const hm_mx_tensor* tensors,
                                          int n, void* stream) {
    if (n < 0 || (n > 0 && !tensors)) return HM_ERR_ARG;
    if (n == 0) return HM_OK;
    if (!w || !q || !scales) return HM_ERR_ARG;
    if (!aligned16(w) || !aligned16(q)) return HM_ERR_ALIGN;
    for (int i = 0; i < n; ++i) {
        const hm_mx_tensor& t = tensors[i];
        if (t.rows < 0 || t.k < 0 || t.src_offset < 0 || t.dst_offset < 0 || t.scale_offset < 0) return HM_ERR_ARG;
        if (t.k % HM_MX_BLOCK || t.src_offset % HM_MX_BLOCK || t.dst_offset % HM_MX_BLOCK) return HM_ERR_ALIGN;
    }
    hm_status st = check_arch();
    if (st != HM_OK) return st;
    for (int g0 = 0; g0 < n; g0 += hm::kInlineRanges) {
        RangeArgs ra;
        std::memset(&ra, 0, sizeof(ra));
        int64_t pre = 0;
        for (int i = g0; i < n && i < g0 + hm::kInlineRanges; ++i) {
            const hm_mx_tensor& t = tensors[i];
            const int64_t len = t.rows * t.k;
            if (!len) continue;
            ra.inl[ra.n++] = Range{t.src_offset, t.dst_offset, t.scale_offset * HM_MX_BLOCK, len, pre, 0.f, 0};
            pre += len;
        }
        ra.total = pre;
        if (!ra.n) continue;
        if (hm::launch_requant(ra, w, q, scales, static_cast<cudaStream_t>(stream)) != cudaSuccess)
            return HM_ERR_CUDA;
    }
    return HM_OK;
}

// ============================================================================
// G with 32 x 32 blocks and Tw's scale relayout (EG1; section 4.1)
// ============================================================================
extern "C" hm_status mxfp8_requant_32x32(const hm_chain* chain, const float* w, uint8_t* q, uint8_t* scales,
                                         const hm_mx_tensor* tensors, int n, void* stream) {
    if (n < 0 || (n > 0 && !tensors)) return HM_ERR_ARG;
    if (n == 0) return HM_OK;
    if (!w || !q || !scales) return HM_ERR_ARG;
    if (chain && chain->so > hm::kMaxChainRanks) return HM_ERR_ARG;
    for (int i = 0; i < n; ++i) {
        const hm_mx_tensor& t = tensors[i];
        if (t.rows < 0 || t.k < 0 || t.src_offset < 0 || t.scale_offset < 0) return HM_ERR_ARG;
        if (t.rows % HM_MX_BLOCK || t.k % HM_MX_BLOCK || t.src_offset % HM_MX_BLOCK) return HM_ERR_ALIGN;
        if (chain && t.src_offset + t.rows * t.k > chain->n) return HM_ERR_GEOMETRY;
    }
    hm_status st = check_arch();
    if (st != HM_OK) return st;
    hm::ChainArgs ch;
    std::memset(&ch, 0, sizeof(ch));
    if (chain) {
        ch.so = chain->so;
        for (int c = 0; c <= chain->so; ++c) ch.edges[c] = chain->edges[c];
        for (int c = 0; c < chain->so; ++c) ch.chunk_base[c] = chain->base[chain->owner[c]];
    }
    for (int g0 = 0; g0 < n; g0 += hm::kMaxMx32Tensors) {
        hm::Mx32Args ta;
        std::memset(&ta, 0, sizeof(ta));
        for (int i = g0; i < n && i < g0 + hm::kMaxMx32Tensors; ++i) {
            const hm_mx_tensor& t = tensors[i];
            if (!t.rows || !t.k) continue;
            ta.src[ta.n] = t.src_offset;
            ta.k[ta.n] = t.k;
            ta.scale_off[ta.n] = t.scale_offset;
            ta.block_prefix[ta.n + 1] = ta.block_prefix[ta.n] + (t.rows / 32) * ((t.k + 127) / 128);  // strips
            ta.n++;
        }
        if (!ta.n) continue;
        if (hm::launch_requant_32x32(ch, ta, w, q, scales, static_cast<cudaStream_t>(stream)) != cudaSuccess)
            return HM_ERR_CUDA;
    }
    return HM_OK;
}

extern "C" hm_status mxfp8_scale_relayout(const uint8_t* src, uint8_t* dst, const hm_scale_relayout* items, int n,
                                          void* stream) {
    if (n < 0 || (n > 0 && !items)) return HM_ERR_ARG;
    if (n == 0) return HM_OK;
    if (!src || !dst) return HM_ERR_ARG;
    for (int i = 0; i < n; ++i) {
        const hm_scale_relayout& it = items[i];
        if (it.rows < 0 || it.kb < 0 || it.src_offset < 0 || it.dst_offset < 0) return HM_ERR_ARG;
        if (it.block_rows != 1 && it.block_rows != 32) return HM_ERR_ARG;
        if (it.rows % it.block_rows) return HM_ERR_ALIGN;
    }
    hm_status st = check_arch();
    if (st != HM_OK) return st;
    for (int g0 = 0; g0 < n; g0 += hm::kMaxRelayoutItems) {
        hm::RelayoutArgs ra;
        std::memset(&ra, 0, sizeof(ra));
        for (int i = g0; i < n && i < g0 + hm::kMaxRelayoutItems; ++i) {
            const hm_scale_relayout& it = items[i];
            if (!it.rows || !it.kb) continue;
            ra.src[ra.n] = it.src_offset;
            ra.dst[ra.n] = it.dst_offset;
            ra.rows[ra.n] = it.rows;
            ra.kb[ra.n] = it.kb;
            ra.block_rows[ra.n] = it.block_rows;
            ra.flags[ra.n] = (((reinterpret_cast<uintptr_t>(src) + it.src_offset) % 16 == 0 && it.kb % 16 == 0)
                                  ? hm::kRelayoutSrc16
                                  : 0) |
                             ((reinterpret_cast<uintptr_t>(dst) + it.dst_offset) % 16 == 0 ? hm::kRelayoutDst16 : 0);
            ra.work_prefix[ra.n + 1] = ra.work_prefix[ra.n] + ((it.rows + 127) / 128) * ((it.kb + 159) / 160);
            ra.n++;
        }
        if (!ra.n) continue;
        if (hm::launch_scale_relayout(ra, src, dst, static_cast<cudaStream_t>(stream)) != cudaSuccess)
            return HM_ERR_CUDA;
    }
    return HM_OK;
}

// ============================================================================
// Outer reduce-scatter of the gradient (sections 3.4 and 4.3; Table 4)
// ============================================================================
extern "C" hm_status reduce_scatter_grad(const hm_chain* chain, const float* parts, int n_parts, int ranks_per_node,
                                         float* g, int mode, int accumulate, uint64_t seed, uint64_t offset,
                                         void* stream) {
    if (!chain || n_parts < 1 || ranks_per_node < 1) return HM_ERR_ARG;
    if (mode < HM_RS_FP32 || mode > HM_RS_BF16_SR) return HM_ERR_ARG;
    if (n_parts % ranks_per_node) return HM_ERR_GEOMETRY;
    if (chain->n == 0) return HM_OK;
    if (!parts || !g) return HM_ERR_ARG;
    if (!aligned16(parts) || !aligned16(g)) return HM_ERR_ALIGN;
    hm_status st = check_arch();
    if (st != HM_OK) return st;
    hm::RsArgs a{};
    a.parts = parts;
    a.stride = chain->n;
    a.n_parts = n_parts;
    a.ranks_per_node = ranks_per_node;
    a.mode = mode;
    a.accumulate = accumulate ? 1 : 0;
    a.seed_lo = static_cast<uint32_t>(seed);
    a.seed_hi = static_cast<uint32_t>(seed >> 32);
    a.offset_lo = static_cast<uint32_t>(offset);
    for (int r0 = 0; r0 < chain->so; r0 += hm::kInlineRanges) {
        RangeArgs ra;
        std::memset(&ra, 0, sizeof(ra));
        int64_t pre = 0;
        for (int r = r0; r < chain->so && r < r0 + hm::kInlineRanges; ++r) {
            if (!chain->len[r]) continue;
            ra.inl[ra.n++] = Range{chain->base[r], chain->edges[chain->chunk_of[r]], 0, chain->len[r], pre, 0.f, 0};
            pre += chain->len[r];
        }
        ra.total = pre;
        if (!ra.n) continue;
        if (hm::launch_reduce_scatter(ra, a, g, static_cast<cudaStream_t>(stream)) != cudaSuccess) return HM_ERR_CUDA;
    }
    return HM_OK;
}
