// Host side of the C ABI declared in include/soma_opt.h.
//
// soma_opt_step: check every argument (nothing changes on failure) -> find
// the list among the handle's prepared lists, else build its norm and update
// tables on the host and upload them -> derive each group's per-step constants in
// fp64 -> enqueue the square-sum kernel, then the update kernel, on the
// caller's stream.  The clip coefficient never leaves the device.
#include "soma_opt.h"

#include <cuda_runtime.h>

#include <algorithm>
#include <array>
#include <cmath>
#include <cstdarg>
#include <cstddef>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <unordered_set>
#include <vector>

#include "soma_kernels.h"

namespace {

// Update chunks: an even number of 8-element vectors per thread of a
// 256-thread CTA.  Lists whose trainable elements mostly have fp32 gradients
// take 8 Ki (four vectors per thread, all covered by the CTA's opening L2
// prefetch); the others 12 Ki (six, the rest covered by the rolling prefetch
// of 16-bit gradients).  Same-box sweep against the earlier 16 Ki: the step
// 1.1 % faster on the flat list and 1.3 % on the 20 000-tensor list (fp32),
// 0.23 % on the 7B shard view and 0.35 % on the action-expert list (bf16);
// odd vector counts per thread (6 Ki, 10 Ki) were up to 8 % slower.
constexpr int32_t kDefaultUpdateChunk = 12288;
constexpr int32_t kDefaultUpdateChunkF32 = 8192;
constexpr int32_t kDefaultNormChunk = 114688;  // 112 Ki: same-box sweeps of 64-192 Ki put it best or within noise
// Norm tables of lists whose owned tensors average at least this many
// elements: larger chunks (less fixed cost per chunk) and a shrinking tail,
// so the last CTAs still end close together.  The chunk that starts with R
// owned elements left holds about R / (kTailShare * resident CTAs), between
// kTailFloor and kLargeNormChunk.  Same-box A/B against 112 Ki: the step
// 0.47 % faster on the action-expert list, 0.11 % on the 7B shard view, 0.07 %
// on the flat list; on the 20 000-tensor list (small tensors) it was slower.
constexpr int32_t kLargeNormChunk = 327680;
constexpr double kTailShare = 0.5;
constexpr int64_t kTailFloor = 32768;
constexpr int64_t kNormCtasPerSm = 3;  // the square-sum kernel's resident CTAs per SM
constexpr int64_t kMinAutoChunk = 1024;   // smallest chunk the automatic sizing picks
constexpr int64_t kUpdateCtasPerSm = 2;   // the update kernel's resident CTAs per SM (its launch bounds)
constexpr int64_t kAutoChunksPerSm = 4;   // small lists: aim for this many chunks per SM
constexpr int64_t kSinglePerCta = 4096;   // default single-launch limit: one 8-element vector per thread of each cluster CTA
constexpr size_t kTimingRing = 1024;
constexpr int kMaxPlans = SOMA_PLAN_CACHE;

struct Group {
    double lr, beta1, beta2, eps, weight_decay;
    int64_t step;
    bool step_dirty;  // the host count is newer than the device table's
    double divisor;   // the group's own effective-batch divisor; 0 = the step's
};

thread_local std::string g_create_error;
std::mutex g_live_mu;
std::unordered_set<const void*> g_live;

bool is_live(const void* h) {
    std::lock_guard<std::mutex> lk(g_live_mu);
    return h != nullptr && g_live.count(h) != 0;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

}  // namespace

// One prepared list: the entries as the caller passed them (the cache key)
// and the device tables and launch shapes built for them.
struct PreparedList {
    bool valid = false;
    uint64_t used = 0;              // stamp of the last step that ran it
    std::vector<soma_tensor_t> key;
    char* d_tables = nullptr;
    size_t cap = 0;                 // bytes
    soma::Table norm_tab{}, upd_tab{};
    std::vector<uint8_t> group_present;
    int norm_grid = 1, upd_grid = 0;
    bool single = false;            // small enough for the single-launch step
    soma_plan_t info{};
};

struct soma_opt {
    int32_t device = 0;
    std::vector<Group> groups;
    std::string err;

    int32_t update_chunk = 0;       // 0: automatic (see chunk_size)
    int32_t norm_chunk = 0;
    int32_t update_ctas_per_sm = 0; // 0: one CTA per chunk
    int32_t norm_ctas_per_sm = 0;
    int64_t single_limit = -1;      // single-launch step up to this many trainable elements; -1: automatic

    // device state, created on first use
    bool dev_ready = false;
    int sm_count = 0;
    int single_ctas = 0;            // CTAs (one cluster) of the single-launch step; 0: not available
    soma::Result* d_res = nullptr;
    soma::Result* h_res = nullptr;  // pinned
    double* d_partials = nullptr;
    size_t partials_cap = 0;        // elements
    char* h_staging = nullptr;      // pinned
    size_t staging_cap = 0;
    cudaEvent_t done = nullptr;     // recorded after each step's last kernel
    bool have_done = false;
    uint32_t nonfinite_read = 0;    // Result::nonfinite_steps at the last soma_opt_get_norm
    void* last_stream = nullptr;
    soma::DevGroup* d_groups = nullptr;  // graph-capturable step: group table
    soma::GroupHp* d_hp = nullptr;       // and the constants of the current step
    float* d_gscale = nullptr;           // group divisors: c / d of each group, per step
    soma::DevGroup* h_groups = nullptr;  // pinned staging of the group table
    cudaEvent_t groups_copied = nullptr; // last copy through h_groups finished
    bool groups_copy_pending = false;
    bool groups_pushed = false;
    bool graph_locked = false;           // a graph step ran: the tables stay as they are

    // Prepared lists, each with its own device tables, so that a step
    // alternating between a few lists (double-buffered gradients, two models
    // on one handle) builds and uploads nothing; the least recently used one
    // is replaced.  Below, copies of the active one's launch parameters.
    std::array<PreparedList, kMaxPlans> plans;
    int active = -1;
    uint64_t stamp = 0;
    int64_t plan_builds = 0, plan_reuses = 0;
    soma::Table norm_tab{}, upd_tab{};
    std::vector<uint8_t> group_present;
    int norm_grid = 1, upd_grid = 0;
    bool single = false;
    soma_plan_t plan{};

    // kernel timing
    bool timing = false;
    std::vector<std::array<cudaEvent_t, 3>> tev;
    size_t tev_used = 0;
    double acc_norm_ms = 0.0, acc_upd_ms = 0.0;
    int64_t acc_steps = 0;

    soma_status_t fail(soma_status_t st, const char* fmt, ...) {
        char buf[512];
        va_list ap;
        va_start(ap, fmt);
        vsnprintf(buf, sizeof buf, fmt, ap);
        va_end(ap);
        err = std::string(soma_status_string(st)) + ": " + buf;
        return st;
    }
    soma_status_t cuda_fail(cudaError_t e, const char* what) {
        cudaGetLastError();  // clear a non-sticky error so later calls start clean
        return fail(e == cudaErrorMemoryAllocation ? SOMA_ERR_OOM : SOMA_ERR_CUDA, "%s: %s (%d)",
                    what, cudaGetErrorString(e), (int)e);
    }
};

namespace {

// Makes `dev` current for the scope and restores the caller's device.
struct DeviceGuard {
    int prev = -1;
    cudaError_t status = cudaSuccess;
    explicit DeviceGuard(int dev) {
        status = cudaGetDevice(&prev);
        if (status == cudaSuccess && prev != dev) status = cudaSetDevice(dev);
    }
    ~DeviceGuard() {
        int cur = -1;
        if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
    }
};

bool is_finite(double x) { return std::isfinite(x); }

soma_status_t check_group_hp(soma_opt* o, double lr, double b1, double b2, double eps, double wd) {
    if (!is_finite(lr) || lr < 0) return o->fail(SOMA_ERR_INVALID_ARG, "lr must be finite and >= 0 (got %g)", lr);
    if (!is_finite(b1) || b1 < 0 || b1 >= 1) return o->fail(SOMA_ERR_INVALID_ARG, "beta1 must be in [0, 1) (got %g)", b1);
    if (!is_finite(b2) || b2 < 0 || b2 >= 1) return o->fail(SOMA_ERR_INVALID_ARG, "beta2 must be in [0, 1) (got %g)", b2);
    if (!is_finite(eps) || eps <= 0) return o->fail(SOMA_ERR_INVALID_ARG, "eps must be finite and > 0 (got %g)", eps);
    if (!is_finite(wd) || wd < 0) return o->fail(SOMA_ERR_INVALID_ARG, "weight_decay must be finite and >= 0 (got %g)", wd);
    return SOMA_OK;
}

int grad_size(uint8_t dtype) { return dtype == SOMA_DTYPE_F32 ? 4 : 2; }

soma_status_t validate_entry(soma_opt* o, const soma_tensor_t& t, int64_t k) {
    if (t.trainable > 1 || t.owned > 1)
        return o->fail(SOMA_ERR_INVALID_ARG, "list[%lld]: trainable and owned must be 0 or 1", (long long)k);
    if (t.numel < 0) return o->fail(SOMA_ERR_INVALID_ARG, "list[%lld].numel < 0", (long long)k);
    if (!t.trainable) return SOMA_OK;
    if (t.group < 0 || t.group >= (int32_t)o->groups.size())
        return o->fail(SOMA_ERR_BAD_GROUP, "list[%lld].group = %d, have %zu groups", (long long)k, t.group,
                       o->groups.size());
    if (t.grad_dtype != SOMA_DTYPE_F32 && t.grad_dtype != SOMA_DTYPE_BF16 && t.grad_dtype != SOMA_DTYPE_F16)
        return o->fail(SOMA_ERR_DTYPE, "list[%lld].grad_dtype = %d", (long long)k, (int)t.grad_dtype);
    // A copy dtype without a copy is an error, except for an empty tensor, whose
    // buffers may all be NULL (an empty torch tensor has no storage).
    if (t.param_lowp ? (t.lowp_dtype != SOMA_DTYPE_BF16 && t.lowp_dtype != SOMA_DTYPE_F16)
                     : (t.lowp_dtype != 0 && t.numel > 0))
        return o->fail(SOMA_ERR_DTYPE, "list[%lld]: lowp_dtype = %d does not match param_lowp", (long long)k,
                       (int)t.lowp_dtype);
    if (t.numel == 0) return SOMA_OK;
    if (!t.param || !t.grad || !t.exp_avg || !t.exp_avg_sq)
        return o->fail(SOMA_ERR_INVALID_ARG, "list[%lld]: null buffer in a trainable entry", (long long)k);
    if ((uintptr_t)t.param % 4 || (uintptr_t)t.exp_avg % 4 || (uintptr_t)t.exp_avg_sq % 4 ||
        (uintptr_t)t.grad % grad_size(t.grad_dtype) || (uintptr_t)t.param_lowp % 2)
        return o->fail(SOMA_ERR_ALIGNMENT, "list[%lld]: a buffer is not aligned to its element size",
                       (long long)k);
    return SOMA_OK;
}

// Head h in [0, 8) of a tensor's vector body: the smallest at which every
// fp32 buffer is 32-byte aligned and every 16-bit one 16-byte aligned (the
// update kernel then moves eight fp32 values per access), else the smallest
// at which every buffer is 16-byte aligned, else -1 (one element at a time).
int vector_head(const uintptr_t* addr, const int* esize, int n) {
    for (int wide = 1; wide >= 0; --wide) {
        for (int h = 0; h < soma::kVec; ++h) {
            bool ok = true;
            for (int k = 0; k < n && ok; ++k) {
                const uintptr_t a = (wide && esize[k] == 4) ? 32 : 16;
                ok = (addr[k] + (uintptr_t)h * esize[k]) % a == 0;
            }
            if (ok) return h;
        }
    }
    return -1;
}

// Cuts tensors into segments and groups segments into chunks of about
// `chunk` elements (at most kMaxSegsPerChunk segments each).
struct TableBuilder {
    int64_t chunk;
    bool one_group_per_chunk;  // norm table: a chunk's partial is scaled by one group's divisor
    std::vector<soma::Seg> segs;
    std::vector<int32_t> begin{0};
    int64_t cur_elems = 0;
    int cur_segs = 0;
    int32_t cur_group = -1;
    // shrinking tail (tail_slots > 0): see kLargeNormChunk
    int64_t tail_total = 0, tail_slots = 0, consumed = 0, cur_target = 0;

    TableBuilder(int64_t c, bool one_group) : chunk(c), one_group_per_chunk(one_group) {}

    // Elements for the chunk that opens now.
    int64_t target() const {
        if (tail_slots <= 0) return chunk;
        const double share = (double)(tail_total - consumed) / (kTailShare * (double)tail_slots);
        return std::max<int64_t>(kTailFloor, std::min<int64_t>(chunk, (int64_t)share / 64 * 64));
    }

    void close() {
        if (cur_segs == 0) return;
        begin.push_back((int32_t)segs.size());
        cur_elems = 0;
        cur_segs = 0;
    }

    // h: vector head of the tensor, -1 = process every element singly.
    void add(const soma_tensor_t& t, int h, bool with_state) {
        const int64_t n = t.numel;
        const int gsz = grad_size(t.grad_dtype);
        int64_t off = 0;
        while (off < n) {
            if (cur_segs == soma::kMaxSegsPerChunk || cur_elems >= cur_target ||
                (one_group_per_chunk && cur_segs > 0 && cur_group != t.group))
                close();
            if (cur_segs == 0) cur_target = target();
            cur_group = t.group;
            const int64_t cut = soma::segment_cut(off, n, cur_target - cur_elems, h);
            const int64_t len = cut - off;
            soma::Seg s{};
            s.p = with_state ? t.param + off : nullptr;
            s.m = with_state ? t.exp_avg + off : nullptr;
            s.v = with_state ? t.exp_avg_sq + off : nullptr;
            s.g = static_cast<const char*>(t.grad) + off * gsz;
            s.plow = (with_state && t.param_lowp) ? static_cast<char*>(t.param_lowp) + off * 2 : nullptr;
            s.lowdt = (with_state && t.param_lowp) ? t.lowp_dtype : 0;
            soma::segment_body(off, len, h, s);
            s.group = (uint16_t)t.group;
            s.gdtype = t.grad_dtype;
            segs.push_back(s);
            cur_elems += len;
            consumed += len;
            ++cur_segs;
            off = cut;
        }
    }
    int32_t nchunks() const { return (int32_t)begin.size() - 1; }
};

soma_status_t ensure_device(soma_opt* o) {
    if (o->dev_ready) return SOMA_OK;
    cudaError_t e;
    if ((e = cudaDeviceGetAttribute(&o->sm_count, cudaDevAttrMultiProcessorCount, o->device)) != cudaSuccess)
        return o->cuda_fail(e, "cudaDeviceGetAttribute");
    o->single_ctas = soma::small_step_cluster_size();
    if ((e = cudaMalloc(&o->d_res, sizeof(soma::Result))) != cudaSuccess) return o->cuda_fail(e, "cudaMalloc(result)");
    if ((e = cudaMemset(o->d_res, 0, sizeof(soma::Result))) != cudaSuccess) return o->cuda_fail(e, "cudaMemset(result)");
    if ((e = cudaMallocHost(&o->h_res, sizeof(soma::Result))) != cudaSuccess) return o->cuda_fail(e, "cudaMallocHost");
    if ((e = cudaEventCreateWithFlags(&o->done, cudaEventDisableTiming)) != cudaSuccess)
        return o->cuda_fail(e, "cudaEventCreate");
    if ((e = cudaMalloc(&o->d_groups, soma::kMaxGroups * sizeof(soma::DevGroup))) != cudaSuccess)
        return o->cuda_fail(e, "cudaMalloc(groups)");
    if ((e = cudaMalloc(&o->d_gscale, soma::kMaxGroups * sizeof(float))) != cudaSuccess)
        return o->cuda_fail(e, "cudaMalloc(group scales)");
    if ((e = cudaMalloc(&o->d_hp, soma::kMaxGroups * sizeof(soma::GroupHp))) != cudaSuccess)
        return o->cuda_fail(e, "cudaMalloc(group constants)");
    if ((e = cudaMemset(o->d_groups, 0, soma::kMaxGroups * sizeof(soma::DevGroup))) != cudaSuccess ||
        (e = cudaMemset(o->d_hp, 0, soma::kMaxGroups * sizeof(soma::GroupHp))) != cudaSuccess)
        return o->cuda_fail(e, "cudaMemset(groups)");
    if ((e = cudaMallocHost(&o->h_groups, soma::kMaxGroups * sizeof(soma::DevGroup))) != cudaSuccess)
        return o->cuda_fail(e, "cudaMallocHost(groups)");
    if ((e = cudaEventCreateWithFlags(&o->groups_copied, cudaEventDisableTiming)) != cudaSuccess)
        return o->cuda_fail(e, "cudaEventCreate");
    o->dev_ready = true;
    return SOMA_OK;
}

// Waits until no kernel of a previous step can still read the tables,
// partials or staging buffer.
soma_status_t wait_idle(soma_opt* o) {
    if (!o->have_done) return SOMA_OK;
    cudaError_t e = cudaEventSynchronize(o->done);
    return e == cudaSuccess ? SOMA_OK : o->cuda_fail(e, "cudaEventSynchronize");
}

// Elements per chunk: the caller's choice, else the default, shrunk for
// lists too small to give every SM a few chunks (down to kMinAutoChunk), so
// that small lists still spread over the whole GPU.
int64_t chunk_size(int32_t requested, int32_t dflt, int64_t total, int sm_count) {
    if (requested > 0) return requested;
    const int64_t spread = (total / (kAutoChunksPerSm * std::max(sm_count, 1)) + 63) / 64 * 64;
    return std::max<int64_t>(kMinAutoChunk, std::min<int64_t>(dflt, spread));
}

// Elements per update chunk.  A list that one wave of the update kernel's
// resident CTAs holds in default chunks is cut into exactly one wave's worth
// of chunks: such lists are latency-bound, and each extra wave adds a CTA's
// fixed cost (tables, the wait for the norm).  Same-box probe, lists of four
// equal tensors, against two waves: 524 Ki elements 10.7 us from 12.4, 1 Mi
// 13.3 from 14.3, 2 Mi 14.7 from 17.5, 3 Mi 18.4 from 19.7 (fp32 gradients
// alike); 256 Ki and smaller unchanged (the 1 Ki floor).  Larger lists keep
// chunk_size's rule.
int64_t update_chunk_size(int32_t requested, int32_t dflt, int64_t total, int sm_count) {
    if (requested > 0) return requested;
    const int64_t slots = kUpdateCtasPerSm * std::max(sm_count, 1);
    if (total <= slots * dflt) {
        const int64_t one_wave = (total + slots - 1) / slots;
        return std::max<int64_t>(kMinAutoChunk, (one_wave + 63) / 64 * 64);
    }
    return chunk_size(requested, dflt, total, sm_count);
}

// Elements per norm chunk of a list whose owned tensors are small on
// average (large ones take kLargeNormChunk): a list that one wave of the
// square-sum kernel's resident CTAs holds in default chunks is cut into one
// wave's worth.  Same-box probe against four chunks per SM: lists of 200,
// 700, 2 700 and 8 000 small tensors (0.7-44 M elements) 3.5-12 % faster
// steps, 1 Mi elements in four tensors 5 %; 256 Ki and smaller unchanged.
int64_t norm_chunk_size(int32_t requested, int32_t dflt, int64_t owned, int sm_count) {
    if (requested > 0) return requested;
    const int64_t slots = kNormCtasPerSm * std::max(sm_count, 1);
    if (owned <= slots * dflt) {
        const int64_t one_wave = (owned + slots - 1) / slots;
        return std::max<int64_t>(kMinAutoChunk, (one_wave + 63) / 64 * 64);
    }
    return chunk_size(requested, dflt, owned, sm_count);
}

// Makes plan i the one the next launches use.
void activate(soma_opt* o, int i) {
    PreparedList& pl = o->plans[i];
    pl.used = ++o->stamp;
    o->active = i;
    o->norm_tab = pl.norm_tab;
    o->upd_tab = pl.upd_tab;
    o->group_present = pl.group_present;
    o->norm_grid = pl.norm_grid;
    o->upd_grid = pl.upd_grid;
    o->single = pl.single;
    o->plan = pl.info;
}

// Index of the prepared list equal to `list`, or -1 (the active one first).
int find_plan(const soma_opt* o, const soma_tensor_t* list, int64_t n) {
    auto equal = [&](const PreparedList& pl) {
        return pl.valid && (int64_t)pl.key.size() == n &&
               (n == 0 || std::memcmp(pl.key.data(), list, (size_t)n * sizeof(soma_tensor_t)) == 0);
    };
    if (o->active >= 0 && equal(o->plans[o->active])) return o->active;
    for (int i = 0; i < kMaxPlans; ++i)
        if (i != o->active && equal(o->plans[i])) return i;
    return -1;
}

// Builds the tables of a list not yet prepared into a free slot, else into
// the least recently used one, and activates it.
soma_status_t rebuild(soma_opt* o, const soma_tensor_t* list, int64_t n, void* stream) {
    int64_t trainable_total = 0, owned_total = 0, owned_tensors = 0, f32_total = 0;
    for (int64_t k = 0; k < n; ++k) {
        if (!list[k].trainable) continue;
        trainable_total += list[k].numel;
        if (list[k].grad_dtype == SOMA_DTYPE_F32) f32_total += list[k].numel;
        if (list[k].owned && list[k].numel > 0) {
            owned_total += list[k].numel;
            owned_tensors += 1;
        }
    }
    // A list for the single-launch step is cut into about one chunk per
    // cluster CTA, so each CTA's share is one pass of its threads.
    const int64_t limit = o->single_limit >= 0 ? o->single_limit : (int64_t)o->single_ctas * kSinglePerCta;
    const bool single = o->single_ctas > 0 && trainable_total <= limit;
    auto per_cta = [&](int64_t total) {  // ceil(total / CTAs), rounded up to a multiple of 64, at least 64
        const int64_t k = std::max(o->single_ctas, 1);
        return std::max<int64_t>(64, ((total + k - 1) / k + 63) / 64 * 64);
    };
    const int32_t upd_default =
        trainable_total > 0 && 2 * f32_total >= trainable_total ? kDefaultUpdateChunkF32 : kDefaultUpdateChunk;
    TableBuilder upd(o->update_chunk == 0 && single
                         ? per_cta(trainable_total)
                         : update_chunk_size(o->update_chunk, upd_default, trainable_total, o->sm_count),
                     false);
    const bool large = o->norm_chunk == 0 && !single && owned_tensors > 0 &&
                       owned_total / owned_tensors >= kLargeNormChunk;
    TableBuilder nrm(o->norm_chunk == 0 && single ? per_cta(owned_total)
                     : large                      ? kLargeNormChunk
                                                  : norm_chunk_size(o->norm_chunk, kDefaultNormChunk, owned_total,
                                                                    o->sm_count), true);
    if (large) {
        nrm.tail_total = owned_total;
        nrm.tail_slots = (int64_t)o->sm_count * kNormCtasPerSm;
    }
    std::vector<uint8_t> present(o->groups.size(), 0);
    int64_t trainable = 0, owned = 0;
    for (int64_t k = 0; k < n; ++k) {
        const soma_tensor_t& t = list[k];
        if (!t.trainable) continue;
        present[t.group] = 1;
        if (t.numel == 0) continue;
        const uintptr_t a5[5] = {(uintptr_t)t.grad, (uintptr_t)t.param, (uintptr_t)t.exp_avg,
                                 (uintptr_t)t.exp_avg_sq, (uintptr_t)t.param_lowp};
        const int e5[5] = {grad_size(t.grad_dtype), 4, 4, 4, 2};
        upd.add(t, vector_head(a5, e5, t.param_lowp ? 5 : 4), true);
        trainable += t.numel;
        if (t.owned) {
            nrm.add(t, vector_head(a5, e5, 1), false);
            owned += t.numel;
        }
    }
    upd.close();
    nrm.close();

    // layout: [update segs][norm segs][update chunk_begin][norm chunk_begin]
    const size_t o_us = 0;
    const size_t o_ns = align_up(o_us + upd.segs.size() * sizeof(soma::Seg), 256);
    const size_t o_ub = align_up(o_ns + nrm.segs.size() * sizeof(soma::Seg), 256);
    const size_t o_nb = align_up(o_ub + upd.begin.size() * sizeof(int32_t), 256);
    const size_t bytes = align_up(o_nb + nrm.begin.size() * sizeof(int32_t), 256);
    const size_t nparts = std::max<size_t>(1, (size_t)nrm.nchunks());

    int slot = 0;
    for (int i = 1; i < kMaxPlans && o->plans[slot].valid; ++i)
        if (!o->plans[i].valid || o->plans[i].used < o->plans[slot].used) slot = i;
    PreparedList& pl = o->plans[slot];

    // a step in flight may still read the slot's tables, the partials or the staging buffer
    soma_status_t st = wait_idle(o);
    if (st != SOMA_OK) return st;
    pl.valid = false;
    if (o->active == slot) o->active = -1;
    cudaError_t e;
    if (bytes > o->staging_cap) {
        if (o->h_staging) cudaFreeHost(o->h_staging);
        o->h_staging = nullptr;
        o->staging_cap = 0;
        if ((e = cudaMallocHost(&o->h_staging, bytes)) != cudaSuccess) return o->cuda_fail(e, "cudaMallocHost(tables)");
        o->staging_cap = bytes;
    }
    if (bytes > pl.cap) {
        if (pl.d_tables) cudaFree(pl.d_tables);
        pl.d_tables = nullptr;
        pl.cap = 0;
        if ((e = cudaMalloc(&pl.d_tables, bytes)) != cudaSuccess) return o->cuda_fail(e, "cudaMalloc(tables)");
        pl.cap = bytes;
    }
    if (nparts > o->partials_cap) {
        if (o->d_partials) cudaFree(o->d_partials);
        o->d_partials = nullptr;
        o->partials_cap = 0;
        if ((e = cudaMalloc(&o->d_partials, nparts * sizeof(double))) != cudaSuccess)
            return o->cuda_fail(e, "cudaMalloc(partials)");
        o->partials_cap = nparts;
    }
    char* h = o->h_staging;
    std::memcpy(h + o_us, upd.segs.data(), upd.segs.size() * sizeof(soma::Seg));
    std::memcpy(h + o_ns, nrm.segs.data(), nrm.segs.size() * sizeof(soma::Seg));
    std::memcpy(h + o_ub, upd.begin.data(), upd.begin.size() * sizeof(int32_t));
    std::memcpy(h + o_nb, nrm.begin.data(), nrm.begin.size() * sizeof(int32_t));
    if ((e = cudaMemcpyAsync(pl.d_tables, h, bytes, cudaMemcpyHostToDevice, (cudaStream_t)stream)) != cudaSuccess)
        return o->cuda_fail(e, "cudaMemcpyAsync(tables)");

    char* d = pl.d_tables;
    pl.upd_tab = soma::Table{reinterpret_cast<const soma::Seg*>(d + o_us),
                             reinterpret_cast<const int32_t*>(d + o_ub), upd.nchunks()};
    pl.norm_tab = soma::Table{reinterpret_cast<const soma::Seg*>(d + o_ns),
                              reinterpret_cast<const int32_t*>(d + o_nb), nrm.nchunks()};
    const int64_t ucap = o->update_ctas_per_sm > 0 ? (int64_t)o->sm_count * o->update_ctas_per_sm : INT32_MAX;
    const int64_t ncap = o->norm_ctas_per_sm > 0 ? (int64_t)o->sm_count * o->norm_ctas_per_sm : INT32_MAX;
    pl.upd_grid = (int)std::min<int64_t>(upd.nchunks(), ucap);
    pl.norm_grid = (int)std::max<int64_t>(1, std::min<int64_t>(nrm.nchunks(), ncap));
    pl.group_present = present;
    pl.single = single;
    pl.key.assign(list, list + n);

    soma_plan_t& p = pl.info;
    p = soma_plan_t{};
    p.norm_chunks = nrm.nchunks();
    p.norm_segments = (int64_t)nrm.segs.size();
    p.update_chunks = upd.nchunks();
    p.update_segments = (int64_t)upd.segs.size();
    p.norm_grid = pl.norm_grid;
    p.norm_block = soma::kNormBlock;
    p.update_grid = pl.upd_grid;
    p.update_block = soma::kUpdateBlock;
    p.trainable_numel = trainable;
    p.owned_numel = owned;
    p.launches_per_step = 1 + (pl.upd_grid > 0 ? 1 : 0);
    pl.valid = true;
    o->plan_builds += 1;
    activate(o, slot);
    return SOMA_OK;
}

soma_status_t timing_flush(soma_opt* o) {
    for (size_t i = 0; i < o->tev_used; ++i) {
        cudaError_t e = cudaEventSynchronize(o->tev[i][2]);
        if (e != cudaSuccess) return o->cuda_fail(e, "cudaEventSynchronize(timing)");
        float a = 0.f, b = 0.f;
        if ((e = cudaEventElapsedTime(&a, o->tev[i][0], o->tev[i][1])) != cudaSuccess ||
            (e = cudaEventElapsedTime(&b, o->tev[i][1], o->tev[i][2])) != cudaSuccess)
            return o->cuda_fail(e, "cudaEventElapsedTime");
        o->acc_norm_ms += a;
        o->acc_upd_ms += b;
        o->acc_steps += 1;
    }
    o->tev_used = 0;
    return SOMA_OK;
}

soma_opt* live_handle(soma_opt_t h) { return is_live(h) ? h : nullptr; }

soma_status_t capturing(soma_opt* o, void* stream, bool* yes) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing((cudaStream_t)stream, &cs);
    if (e != cudaSuccess) return o->cuda_fail(e, "cudaStreamIsCapturing");
    *yes = cs != cudaStreamCaptureStatusNone;
    return SOMA_OK;
}

// The regular and multi-rank steps fix their constants (lr, step counts,
// bias corrections) on the host when they enqueue, and may wait on the host
// for a new list's tables: a captured launch would replay stale constants, so
// they refuse stream capture (soma_opt_step_graph is the capturable step).
soma_status_t refuse_capture(soma_opt* o, void* stream, const char* what) {
    bool cap = false;
    soma_status_t st = capturing(o, stream, &cap);
    if (st != SOMA_OK) return st;
    if (cap)
        return o->fail(SOMA_ERR_STATE, "%s cannot be captured in a CUDA graph (its constants are fixed when it is "
                                       "enqueued); capture soma_opt_step_graph instead", what);
    return SOMA_OK;
}

// Common argument checks of the step entry points.  *hit: the prepared list
// equal to `list`, or -1; only a list not prepared yet is validated entry by
// entry (a prepared one was validated when it was built, and groups are never
// removed).
soma_status_t check_step_args(soma_opt* o, const soma_tensor_t* list, int64_t n, double grad_divisor,
                              double max_norm, int* hit) {
    if (n < 0) return o->fail(SOMA_ERR_INVALID_ARG, "n < 0");
    if (n > 0 && !list) return o->fail(SOMA_ERR_INVALID_ARG, "list is NULL with n > 0");
    if (!is_finite(grad_divisor) || grad_divisor <= 0)
        return o->fail(SOMA_ERR_INVALID_ARG, "grad_divisor must be finite and > 0 (got %g)", grad_divisor);
    if (!is_finite(max_norm) || max_norm <= 0)
        return o->fail(SOMA_ERR_INVALID_ARG, "max_norm must be finite and > 0 (got %g)", max_norm);
    *hit = find_plan(o, list, n);
    if (*hit < 0) {
        for (int64_t k = 0; k < n; ++k) {
            soma_status_t st = validate_entry(o, list[k], k);
            if (st != SOMA_OK) return st;
        }
    }
    return SOMA_OK;
}

}  // namespace

extern "C" {

const char* soma_status_string(soma_status_t s) {
    switch (s) {
        case SOMA_OK: return "ok";
        case SOMA_ERR_INVALID_ARG: return "invalid argument";
        case SOMA_ERR_BAD_GROUP: return "unknown parameter group";
        case SOMA_ERR_DTYPE: return "unsupported gradient dtype";
        case SOMA_ERR_ALIGNMENT: return "misaligned buffer";
        case SOMA_ERR_OOM: return "out of memory";
        case SOMA_ERR_CUDA: return "CUDA error";
        case SOMA_ERR_STATE: return "invalid handle or state";
        case SOMA_ERR_LIMIT: return "limit exceeded";
        default: return "unknown status";
    }
}

int32_t soma_abi_version(void) { return SOMA_ABI_VERSION; }

soma_status_t soma_opt_create(soma_opt_t* out, int32_t device) {
    if (!out) {
        g_create_error = "invalid argument: out is NULL";
        return SOMA_ERR_INVALID_ARG;
    }
    *out = nullptr;
    if (device < 0) {
        g_create_error = "invalid argument: device < 0";
        return SOMA_ERR_INVALID_ARG;
    }
    soma_opt* o = new (std::nothrow) soma_opt();
    if (!o) {
        g_create_error = "out of memory: handle";
        return SOMA_ERR_OOM;
    }
    o->device = device;
    {
        std::lock_guard<std::mutex> lk(g_live_mu);
        g_live.insert(o);
    }
    *out = o;
    return SOMA_OK;
}

const char* soma_opt_last_error(soma_opt_t h) {
    if (h == nullptr) return g_create_error.c_str();
    soma_opt* o = live_handle(h);
    return o ? o->err.c_str() : "invalid handle";
}

soma_status_t soma_opt_add_group(soma_opt_t h, double lr, double beta1, double beta2, double eps,
                                 double weight_decay, int32_t* group_id) {
    soma_opt* o = live_handle(h);
    if (!o) return SOMA_ERR_STATE;
    if (!group_id) return o->fail(SOMA_ERR_INVALID_ARG, "group_id is NULL");
    soma_status_t st = check_group_hp(o, lr, beta1, beta2, eps, weight_decay);
    if (st != SOMA_OK) return st;
    if ((int)o->groups.size() >= SOMA_MAX_GROUPS)
        return o->fail(SOMA_ERR_LIMIT, "at most %d parameter groups", SOMA_MAX_GROUPS);
    o->groups.push_back(Group{lr, beta1, beta2, eps, weight_decay, 0, true, 0.0});
    *group_id = (int32_t)o->groups.size() - 1;
    return SOMA_OK;
}

soma_status_t soma_opt_set_lr(soma_opt_t h, int32_t group, double lr) {
    soma_opt* o = live_handle(h);
    if (!o) return SOMA_ERR_STATE;
    if (group < 0 || group >= (int32_t)o->groups.size()) return o->fail(SOMA_ERR_BAD_GROUP, "group %d", group);
    if (!is_finite(lr) || lr < 0) return o->fail(SOMA_ERR_INVALID_ARG, "lr must be finite and >= 0 (got %g)", lr);
    o->groups[group].lr = lr;
    return SOMA_OK;
}

soma_status_t soma_opt_get_group(soma_opt_t h, int32_t group, double* lr, double* beta1, double* beta2,
                                 double* eps, double* weight_decay) {
    soma_opt* o = live_handle(h);
    if (!o) return SOMA_ERR_STATE;
    if (group < 0 || group >= (int32_t)o->groups.size()) return o->fail(SOMA_ERR_BAD_GROUP, "group %d", group);
    const Group& g = o->groups[group];
    if (lr) *lr = g.lr;
    if (beta1) *beta1 = g.beta1;
    if (beta2) *beta2 = g.beta2;
    if (eps) *eps = g.eps;
    if (weight_decay) *weight_decay = g.weight_decay;
    return SOMA_OK;
}

soma_status_t soma_opt_set_group(soma_opt_t h, int32_t group, double lr, double beta1, double beta2,
                                 double eps, double weight_decay) {
    soma_opt* o = live_handle(h);
    if (!o) return SOMA_ERR_STATE;
    if (group < 0 || group >= (int32_t)o->groups.size()) return o->fail(SOMA_ERR_BAD_GROUP, "group %d", group);
    soma_status_t st = check_group_hp(o, lr, beta1, beta2, eps, weight_decay);
    if (st != SOMA_OK) return st;
    Group& g = o->groups[group];
    g.lr = lr;
    g.beta1 = beta1;
    g.beta2 = beta2;
    g.eps = eps;
    g.weight_decay = weight_decay;
    return SOMA_OK;
}

soma_status_t soma_opt_set_group_divisor(soma_opt_t h, int32_t group, double divisor) {
    soma_opt* o = live_handle(h);
    if (!o) return SOMA_ERR_STATE;
    if (group < 0 || group >= (int32_t)o->groups.size()) return o->fail(SOMA_ERR_BAD_GROUP, "group %d", group);
    if (!is_finite(divisor) || divisor < 0)
        return o->fail(SOMA_ERR_INVALID_ARG, "divisor must be finite and >= 0 (got %g)", divisor);
    o->groups[group].divisor = divisor;
    return SOMA_OK;
}

soma_status_t soma_opt_get_group_divisor(soma_opt_t h, int32_t group, double* divisor) {
    soma_opt* o = live_handle(h);
    if (!o) return SOMA_ERR_STATE;
    if (group < 0 || group >= (int32_t)o->groups.size()) return o->fail(SOMA_ERR_BAD_GROUP, "group %d", group);
    if (!divisor) return o->fail(SOMA_ERR_INVALID_ARG, "divisor is NULL");
    *divisor = o->groups[group].divisor;
    return SOMA_OK;
}

soma_status_t soma_opt_get_group_step(soma_opt_t h, int32_t group, int64_t* t) {
    soma_opt* o = live_handle(h);
    if (!o) return SOMA_ERR_STATE;
    if (group < 0 || group >= (int32_t)o->groups.size()) return o->fail(SOMA_ERR_BAD_GROUP, "group %d", group);
    if (!t) return o->fail(SOMA_ERR_INVALID_ARG, "t is NULL");
    *t = o->groups[group].step;
    return SOMA_OK;
}

soma_status_t soma_opt_set_group_step(soma_opt_t h, int32_t group, int64_t t) {
    soma_opt* o = live_handle(h);
    if (!o) return SOMA_ERR_STATE;
    if (group < 0 || group >= (int32_t)o->groups.size()) return o->fail(SOMA_ERR_BAD_GROUP, "group %d", group);
    if (t < 0) return o->fail(SOMA_ERR_INVALID_ARG, "step count must be >= 0");
    o->groups[group].step = t;
    o->groups[group].step_dirty = true;
    return SOMA_OK;
}

soma_status_t soma_opt_set_tuning(soma_opt_t h, int32_t update_chunk, int32_t norm_chunk,
                                  int32_t update_ctas_per_sm, int32_t norm_ctas_per_sm) {
    soma_opt* o = live_handle(h);
    if (!o) return SOMA_ERR_STATE;
    auto ok_chunk = [](int32_t c) { return c == 0 || (c >= 64 && c <= (1 << 26)); };
    if (!ok_chunk(update_chunk) || !ok_chunk(norm_chunk))
        return o->fail(SOMA_ERR_INVALID_ARG, "chunk sizes must be 0 or in [64, 2^26]");
    if (update_ctas_per_sm < 0 || update_ctas_per_sm > 64 || norm_ctas_per_sm < 0 || norm_ctas_per_sm > 64)
        return o->fail(SOMA_ERR_INVALID_ARG, "CTAs per SM must be in [0, 64]");
    if (o->graph_locked) return o->fail(SOMA_ERR_STATE, "this handle ran a graph-capturable step: its plan is fixed");
    o->update_chunk = update_chunk / 64 * 64;
    o->norm_chunk = norm_chunk / 64 * 64;
    o->update_ctas_per_sm = update_ctas_per_sm;
    o->norm_ctas_per_sm = norm_ctas_per_sm;
    for (auto& pl : o->plans) pl.valid = false;
    o->active = -1;
    return SOMA_OK;
}

soma_status_t soma_opt_set_single_launch(soma_opt_t h, int64_t max_elements) {
    soma_opt* o = live_handle(h);
    if (!o) return SOMA_ERR_STATE;
    if (max_elements < -1) return o->fail(SOMA_ERR_INVALID_ARG, "max_elements must be -1, 0 or positive");
    if (o->graph_locked) return o->fail(SOMA_ERR_STATE, "this handle ran a graph-capturable step: its plan is fixed");
    o->single_limit = max_elements;
    for (auto& pl : o->plans) pl.valid = false;
    o->active = -1;
    return SOMA_OK;
}

namespace {

// Does a group present in the active list set its own divisor?
bool any_group_divisor(const soma_opt* o) {
    for (size_t q = 0; q < o->groups.size(); ++q)
        if (o->groups[q].divisor > 0 && q < o->group_present.size() && o->group_present[q]) return true;
    return false;
}

// 1 / (effective divisor) of every group, its own or else the step's: the
// square-sum scales each chunk partial by its square, and c times it is the
// group's update scale.
void fill_divisors(const soma_opt* o, double grad_divisor, double* inv) {
    for (int q = 0; q < soma::kMaxGroups; ++q) {
        const double d = (q < (int)o->groups.size() && o->groups[q].divisor > 0) ? o->groups[q].divisor
                                                                                 : grad_divisor;
        inv[q] = 1.0 / d;
    }
}

// Everything a step does before its launches, after the arguments were
// checked: device, ordering after the previous step, tables for this list.
soma_status_t prepare(soma_opt* o, const soma_tensor_t* list, int64_t n, int hit, void* stream) {
    soma_status_t st = ensure_device(o);
    if (st != SOMA_OK) return st;
    cudaError_t e;
    if (o->have_done && o->last_stream != stream) {
        // order this step after the previous one, whatever stream that ran on
        if ((e = cudaStreamWaitEvent((cudaStream_t)stream, o->done, 0)) != cudaSuccess)
            return o->cuda_fail(e, "cudaStreamWaitEvent");
    }
    if (hit >= 0) {
        activate(o, hit);
        o->plan_reuses += 1;
        return SOMA_OK;
    }
    return rebuild(o, list, n, stream);
}

// Per-group constants of the next step (fp64, rounded once; the graph step
// derives the same bits on the device) and the step counts it will reach.
void host_group_constants(soma_opt* o, soma::UpdateArgs& ua, std::vector<int64_t>& next) {
    next.assign(o->groups.size(), 0);
    for (size_t q = 0; q < o->groups.size(); ++q) {
        const Group& g = o->groups[q];
        const bool on = q < o->group_present.size() && o->group_present[q];
        next[q] = g.step + (on ? 1 : 0);
        if (!on) continue;
        ua.groups[q] = soma::make_group_hp(g.lr, g.beta1, g.beta2, g.eps, g.weight_decay, next[q]);
    }
}

// The launches of a step: the norm side (the square-sum kernel, or for the
// multi-rank step the finish kernel over the ranks' sums), then the update.
soma_status_t launch_step(soma_opt* o, double grad_divisor, double max_norm, const double* rank_sums,
                          int32_t nranks, void* stream) {
    soma::UpdateArgs ua{};
    ua.t = o->upd_tab;
    ua.res = o->d_res;
    ua.ngroups = (int32_t)o->groups.size();
    ua.gscale = o->d_gscale;
    std::vector<int64_t> next;
    host_group_constants(o, ua, next);
    cudaError_t e;
    soma_status_t st;
    bool single = false;
    std::array<cudaEvent_t, 3>* ev = nullptr;
    if (o->timing) {
        if (o->tev_used == kTimingRing && (st = timing_flush(o)) != SOMA_OK) return st;
        if (o->tev_used == o->tev.size()) {
            std::array<cudaEvent_t, 3> t3{};
            for (auto& x : t3)
                if ((e = cudaEventCreate(&x)) != cudaSuccess) return o->cuda_fail(e, "cudaEventCreate(timing)");
            o->tev.push_back(t3);
        }
        ev = &o->tev[o->tev_used];
        if ((e = cudaEventRecord((*ev)[0], (cudaStream_t)stream)) != cudaSuccess)
            return o->cuda_fail(e, "cudaEventRecord");
    }
    if (rank_sums) {
        soma::FinishArgs fa{};
        fa.parts = rank_sums;
        fa.count = nranks;
        fa.res = o->d_res;
        fa.divisor = grad_divisor;
        fa.inv_step_divisor = 1.0 / grad_divisor;
        fa.max_norm = max_norm;
        if (any_group_divisor(o)) {
            fa.gscale = o->d_gscale;
            fa.ngroups = (int32_t)o->groups.size();
            fill_divisors(o, grad_divisor, fa.inv_divisor);
        }
        if ((e = (cudaError_t)soma::launch_finish(fa, stream)) != cudaSuccess)
            return o->cuda_fail(e, "launching the finish kernel");
    } else {
        soma::NormArgs na{};
        na.t = o->norm_tab;
        na.partials = o->d_partials;
        na.res = o->d_res;
        na.divisor = grad_divisor;
        na.inv_step_divisor = 1.0 / grad_divisor;
        na.max_norm = max_norm;
        fill_divisors(o, grad_divisor, na.inv_divisor);
        na.gscale = o->d_gscale;
        na.ngroups = (int32_t)o->groups.size();
        // Small lists run as one launch, unless timing events must separate
        // the two kernels.
        single = o->single && ev == nullptr;
        if (single) {
            if ((e = (cudaError_t)soma::launch_small_step(na, ua, o->single_ctas, stream, true, false,
                                                          any_group_divisor(o))) != cudaSuccess)
                return o->cuda_fail(e, "launching the single-launch step");
        } else if ((e = (cudaError_t)soma::launch_norm(na, o->norm_grid, stream, false, any_group_divisor(o),
                                                       ev == nullptr)) != cudaSuccess) {
            return o->cuda_fail(e, "launching the square-sum kernel");
        }
    }
    if (ev && (e = cudaEventRecord((*ev)[1], (cudaStream_t)stream)) != cudaSuccess)
        return o->cuda_fail(e, "cudaEventRecord");
    // without a timing event between the two kernels, the update kernel may
    // overlap the square-sum kernel's tail
    if (!single && o->upd_grid > 0 &&
        (e = (cudaError_t)soma::launch_update(ua, o->upd_grid, stream, false, ev == nullptr,
                                              any_group_divisor(o))) != cudaSuccess)
        return o->cuda_fail(e, "launching the update kernel");
    o->plan.launches_per_step = single ? 1 : 1 + (o->upd_grid > 0 ? 1 : 0);
    o->plan.single_launch_ctas = single ? o->single_ctas : 0;
    if (ev) {
        if ((e = cudaEventRecord((*ev)[2], (cudaStream_t)stream)) != cudaSuccess)
            return o->cuda_fail(e, "cudaEventRecord");
        o->tev_used += 1;
    }
    if ((e = cudaEventRecord(o->done, (cudaStream_t)stream)) != cudaSuccess)
        return o->cuda_fail(e, "cudaEventRecord");
    o->have_done = true;
    o->last_stream = stream;
    for (size_t q = 0; q < o->groups.size(); ++q) {
        if (next[q] != o->groups[q].step) o->groups[q].step_dirty = true;
        o->groups[q].step = next[q];
    }
    return SOMA_OK;
}

}  // namespace

soma_status_t soma_opt_step(soma_opt_t h, const soma_tensor_t* list, int64_t n, double grad_divisor,
                            double max_norm, void* stream) {
    soma_opt* o = live_handle(h);
    if (!o) return SOMA_ERR_STATE;
    int hit = -1;
    soma_status_t st = check_step_args(o, list, n, grad_divisor, max_norm, &hit);
    if (st != SOMA_OK) return st;
    if (o->graph_locked && hit != o->active)
        return o->fail(SOMA_ERR_STATE, "this handle ran a graph-capturable step: it keeps that list");
    DeviceGuard dg(o->device);
    if (dg.status != cudaSuccess) return o->cuda_fail(dg.status, "selecting the device");
    if ((st = refuse_capture(o, stream, "soma_opt_step")) != SOMA_OK) return st;
    if ((st = prepare(o, list, n, hit, stream)) != SOMA_OK) return st;
    return launch_step(o, grad_divisor, max_norm, nullptr, 0, stream);
}

soma_status_t soma_opt_sumsq(soma_opt_t h, const soma_tensor_t* list, int64_t n, double grad_divisor,
                             double* sumsq_out, void* stream) {
    soma_opt* o = live_handle(h);
    if (!o) return SOMA_ERR_STATE;
    if (!sumsq_out || (uintptr_t)sumsq_out % alignof(double) != 0)
        return o->fail(SOMA_ERR_INVALID_ARG, "sumsq_out must be a non-null, 8-byte aligned device pointer");
    int hit = -1;
    soma_status_t st = check_step_args(o, list, n, grad_divisor, 1.0, &hit);
    if (st != SOMA_OK) return st;
    if (o->graph_locked && hit != o->active)
        return o->fail(SOMA_ERR_STATE, "this handle ran a graph-capturable step: it keeps that list");
    DeviceGuard dg(o->device);
    if (dg.status != cudaSuccess) return o->cuda_fail(dg.status, "selecting the device");
    if ((st = refuse_capture(o, stream, "soma_opt_sumsq")) != SOMA_OK) return st;
    if ((st = prepare(o, list, n, hit, stream)) != SOMA_OK) return st;
    soma::NormArgs na{};
    na.t = o->norm_tab;
    na.partials = o->d_partials;
    na.res = o->d_res;
    na.divisor = grad_divisor;
    na.inv_step_divisor = 1.0 / grad_divisor;
    na.max_norm = 1.0;
    na.sumsq_out = sumsq_out;
    fill_divisors(o, grad_divisor, na.inv_divisor);
    na.gscale = o->d_gscale;
    na.ngroups = (int32_t)o->groups.size();
    cudaError_t e;
    if ((e = (cudaError_t)soma::launch_norm(na, o->norm_grid, stream, false, any_group_divisor(o), true)) !=
        cudaSuccess)
        return o->cuda_fail(e, "launching the square-sum kernel");
    if ((e = cudaEventRecord(o->done, (cudaStream_t)stream)) != cudaSuccess)
        return o->cuda_fail(e, "cudaEventRecord");
    o->have_done = true;
    o->last_stream = stream;
    return SOMA_OK;
}

soma_status_t soma_opt_step_from_sumsq(soma_opt_t h, const soma_tensor_t* list, int64_t n, double grad_divisor,
                                       double max_norm, const double* rank_sumsq, int32_t nranks,
                                       void* stream) {
    soma_opt* o = live_handle(h);
    if (!o) return SOMA_ERR_STATE;
    if (!rank_sumsq || (uintptr_t)rank_sumsq % alignof(double) != 0)
        return o->fail(SOMA_ERR_INVALID_ARG, "rank_sumsq must be a non-null, 8-byte aligned device pointer");
    if (nranks < 1 || nranks > SOMA_MAX_RANKS)
        return o->fail(SOMA_ERR_INVALID_ARG, "nranks must be in [1, %d]", SOMA_MAX_RANKS);
    int hit = -1;
    soma_status_t st = check_step_args(o, list, n, grad_divisor, max_norm, &hit);
    if (st != SOMA_OK) return st;
    if (o->graph_locked && hit != o->active)
        return o->fail(SOMA_ERR_STATE, "this handle ran a graph-capturable step: it keeps that list");
    DeviceGuard dg(o->device);
    if (dg.status != cudaSuccess) return o->cuda_fail(dg.status, "selecting the device");
    if ((st = refuse_capture(o, stream, "soma_opt_step_from_sumsq")) != SOMA_OK) return st;
    if ((st = prepare(o, list, n, hit, stream)) != SOMA_OK) return st;
    return launch_step(o, grad_divisor, max_norm, rank_sumsq, nranks, stream);
}

soma_status_t soma_opt_step_graph(soma_opt_t h, const soma_tensor_t* list, int64_t n, double grad_divisor,
                                  double max_norm, void* stream) {
    soma_opt* o = live_handle(h);
    if (!o) return SOMA_ERR_STATE;
    int hit = -1;
    soma_status_t st = check_step_args(o, list, n, grad_divisor, max_norm, &hit);
    if (st != SOMA_OK) return st;
    if (o->graph_locked && hit != o->active)
        return o->fail(SOMA_ERR_STATE, "this handle ran a graph-capturable step: it keeps that list");
    DeviceGuard dg(o->device);
    if (dg.status != cudaSuccess) return o->cuda_fail(dg.status, "selecting the device");
    bool cap = false;
    if ((st = capturing(o, stream, &cap)) != SOMA_OK) return st;
    if (cap && (!o->dev_ready || hit < 0 || hit != o->active))
        return o->fail(SOMA_ERR_STATE, "run soma_opt_step_graph once with this list before capturing it");
    if (!o->groups_pushed)
        return o->fail(SOMA_ERR_STATE, "soma_opt_push_groups must run before the first graph-capturable step");
    if ((st = ensure_device(o)) != SOMA_OK) return st;
    cudaError_t e;
    if (!cap && o->have_done && o->last_stream != stream &&
        (e = cudaStreamWaitEvent((cudaStream_t)stream, o->done, 0)) != cudaSuccess)
        return o->cuda_fail(e, "cudaStreamWaitEvent");
    if (hit >= 0) {
        activate(o, hit);
        o->plan_reuses += 1;
    } else if ((st = rebuild(o, list, n, stream)) != SOMA_OK) {
        return st;
    }
    uint64_t present = 0;
    for (size_t q = 0; q < o->group_present.size(); ++q)
        if (o->group_present[q]) present |= 1ull << q;
    soma::NormArgs na{};
    na.t = o->norm_tab;
    na.partials = o->d_partials;
    na.res = o->d_res;
    na.divisor = grad_divisor;
    na.inv_step_divisor = 1.0 / grad_divisor;
    na.max_norm = max_norm;
    na.dgroups = o->d_groups;
    na.dhp = o->d_hp;
    na.present = present;
    na.ngroups = (int32_t)o->groups.size();
    na.gscale = o->d_gscale;
    fill_divisors(o, grad_divisor, na.inv_divisor);
    soma::UpdateArgs ua{};
    ua.t = o->upd_tab;
    ua.res = o->d_res;
    ua.dhp = o->d_hp;
    ua.ngroups = (int32_t)o->groups.size();
    ua.gscale = o->d_gscale;
    const bool single = o->single;
    if (single) {
        if ((e = (cudaError_t)soma::launch_small_step(na, ua, o->single_ctas, stream, true, true,
                                                      any_group_divisor(o))) != cudaSuccess)
            return o->cuda_fail(e, "launching the single-launch step");
    } else {
        // one CTA more than the chunks need: CTA 0 derives the group constants
        if ((e = (cudaError_t)soma::launch_norm(na, o->norm_grid + 1, stream, true, any_group_divisor(o))) !=
            cudaSuccess)
            return o->cuda_fail(e, "launching the square-sum kernel");
        if (o->upd_grid > 0 &&
            (e = (cudaError_t)soma::launch_update(ua, o->upd_grid, stream, true, true, any_group_divisor(o))) !=
                cudaSuccess)
            return o->cuda_fail(e, "launching the update kernel");
    }
    o->plan.launches_per_step = single ? 1 : 1 + (o->upd_grid > 0 ? 1 : 0);
    o->plan.single_launch_ctas = single ? o->single_ctas : 0;
    o->graph_locked = true;
    if (!cap) {
        if ((e = cudaEventRecord(o->done, (cudaStream_t)stream)) != cudaSuccess)
            return o->cuda_fail(e, "cudaEventRecord");
        o->have_done = true;
        o->last_stream = stream;
    }
    return SOMA_OK;
}

soma_status_t soma_opt_push_groups(soma_opt_t h, void* stream) {
    soma_opt* o = live_handle(h);
    if (!o) return SOMA_ERR_STATE;
    DeviceGuard dg(o->device);
    if (dg.status != cudaSuccess) return o->cuda_fail(dg.status, "selecting the device");
    bool cap = false;
    soma_status_t st = capturing(o, stream, &cap);
    if (st != SOMA_OK) return st;
    if (cap) return o->fail(SOMA_ERR_STATE, "soma_opt_push_groups cannot be captured");
    if ((st = ensure_device(o)) != SOMA_OK) return st;
    // The copy engine reads the staging buffer when the copy runs, not when it
    // is enqueued: wait until the previous copy through it has finished.
    cudaError_t e;
    if (o->groups_copy_pending && (e = cudaEventSynchronize(o->groups_copied)) != cudaSuccess)
        return o->cuda_fail(e, "cudaEventSynchronize(groups)");
    o->groups_copy_pending = false;
    const size_t ng = o->groups.size();
    for (size_t q = 0; q < ng; ++q) {
        const Group& g = o->groups[q];
        o->h_groups[q] = soma::DevGroup{g.lr, g.beta1, g.beta2, g.eps, g.weight_decay, g.step, {0, 0}};
    }
    if (ng > 0) {
        // hyperparameters: the first 40 bytes of every 64-byte entry
        const size_t hp_bytes = offsetof(soma::DevGroup, step);
        if ((e = cudaMemcpy2DAsync(o->d_groups, sizeof(soma::DevGroup), o->h_groups, sizeof(soma::DevGroup),
                                   hp_bytes, ng, cudaMemcpyHostToDevice, (cudaStream_t)stream)) != cudaSuccess)
            return o->cuda_fail(e, "cudaMemcpy2DAsync(groups)");
        // step counts only where the host count is newer (first push,
        // soma_opt_set_group_step, regular steps): graph steps advance the
        // device count and must not be rolled back
        for (size_t q = 0; q < ng; ++q) {
            if (!o->groups[q].step_dirty) continue;
            if ((e = cudaMemcpyAsync(&o->d_groups[q].step, &o->h_groups[q].step, sizeof(int64_t),
                                     cudaMemcpyHostToDevice, (cudaStream_t)stream)) != cudaSuccess)
                return o->cuda_fail(e, "cudaMemcpyAsync(group step)");
            o->groups[q].step_dirty = false;
        }
        if ((e = cudaEventRecord(o->groups_copied, (cudaStream_t)stream)) != cudaSuccess)
            return o->cuda_fail(e, "cudaEventRecord(groups)");
        o->groups_copy_pending = true;
    }
    o->groups_pushed = true;
    return SOMA_OK;
}

soma_status_t soma_opt_pull_groups(soma_opt_t h, void* stream) {
    soma_opt* o = live_handle(h);
    if (!o) return SOMA_ERR_STATE;
    if (!o->groups_pushed) return o->fail(SOMA_ERR_STATE, "no group table on the device yet");
    DeviceGuard dg(o->device);
    if (dg.status != cudaSuccess) return o->cuda_fail(dg.status, "selecting the device");
    bool cap = false;
    soma_status_t st = capturing(o, stream, &cap);
    if (st != SOMA_OK) return st;
    if (cap) return o->fail(SOMA_ERR_STATE, "soma_opt_pull_groups cannot be captured");
    cudaError_t e;
    if (o->groups_copy_pending && (e = cudaEventSynchronize(o->groups_copied)) != cudaSuccess)
        return o->cuda_fail(e, "cudaEventSynchronize(groups)");
    o->groups_copy_pending = false;
    const size_t ng = o->groups.size();
    if (ng > 0 && (e = cudaMemcpyAsync(o->h_groups, o->d_groups, ng * sizeof(soma::DevGroup),
                                       cudaMemcpyDeviceToHost, (cudaStream_t)stream)) != cudaSuccess)
        return o->cuda_fail(e, "cudaMemcpyAsync(groups)");
    if ((e = cudaStreamSynchronize((cudaStream_t)stream)) != cudaSuccess)
        return o->cuda_fail(e, "cudaStreamSynchronize");
    for (size_t q = 0; q < ng; ++q) {
        o->groups[q].step = o->h_groups[q].step;
        o->groups[q].step_dirty = false;
    }
    return SOMA_OK;
}

soma_status_t soma_opt_device_groups(soma_opt_t h, soma_device_group_t** table) {
    soma_opt* o = live_handle(h);
    if (!o) return SOMA_ERR_STATE;
    if (!table) return o->fail(SOMA_ERR_INVALID_ARG, "table is NULL");
    DeviceGuard dg(o->device);
    if (dg.status != cudaSuccess) return o->cuda_fail(dg.status, "selecting the device");
    soma_status_t st = ensure_device(o);
    if (st != SOMA_OK) return st;
    *table = reinterpret_cast<soma_device_group_t*>(o->d_groups);
    return SOMA_OK;
}

soma_status_t soma_opt_get_norm(soma_opt_t h, double* norm, double* clip_coef, int32_t* nonfinite, void* stream) {
    soma_opt* o = live_handle(h);
    if (!o) return SOMA_ERR_STATE;
    if (!o->have_done) return o->fail(SOMA_ERR_STATE, "no step has run on this handle");
    DeviceGuard dg(o->device);
    if (dg.status != cudaSuccess) return o->cuda_fail(dg.status, "selecting the device");
    cudaError_t e;
    if (o->last_stream != stream && (e = cudaStreamWaitEvent((cudaStream_t)stream, o->done, 0)) != cudaSuccess)
        return o->cuda_fail(e, "cudaStreamWaitEvent");
    if ((e = cudaMemcpyAsync(o->h_res, o->d_res, sizeof(soma::Result), cudaMemcpyDeviceToHost,
                             (cudaStream_t)stream)) != cudaSuccess)
        return o->cuda_fail(e, "cudaMemcpyAsync(result)");
    if ((e = cudaStreamSynchronize((cudaStream_t)stream)) != cudaSuccess)
        return o->cuda_fail(e, "cudaStreamSynchronize");
    if (norm) *norm = o->h_res->norm;
    if (clip_coef) *clip_coef = o->h_res->coef;
    // the device count only grows; report the steps since the previous read
    const uint32_t seen = o->h_res->nonfinite_steps;
    if (nonfinite) *nonfinite = (int32_t)std::min<uint32_t>(seen - o->nonfinite_read, INT32_MAX);
    o->nonfinite_read = seen;
    return SOMA_OK;
}

soma_status_t soma_opt_set_timing(soma_opt_t h, int32_t enable) {
    soma_opt* o = live_handle(h);
    if (!o) return SOMA_ERR_STATE;
    if (enable != 0 && enable != 1) return o->fail(SOMA_ERR_INVALID_ARG, "enable must be 0 or 1");
    o->timing = enable != 0;
    return SOMA_OK;
}

soma_status_t soma_opt_read_timing(soma_opt_t h, double* norm_ms, double* update_ms, int64_t* steps) {
    soma_opt* o = live_handle(h);
    if (!o) return SOMA_ERR_STATE;
    if (o->tev_used) {
        DeviceGuard dg(o->device);
        if (dg.status != cudaSuccess) return o->cuda_fail(dg.status, "selecting the device");
        soma_status_t st = timing_flush(o);
        if (st != SOMA_OK) return st;
    }
    if (norm_ms) *norm_ms = o->acc_norm_ms;
    if (update_ms) *update_ms = o->acc_upd_ms;
    if (steps) *steps = o->acc_steps;
    o->acc_norm_ms = o->acc_upd_ms = 0.0;
    o->acc_steps = 0;
    return SOMA_OK;
}

soma_status_t soma_opt_get_plan(soma_opt_t h, soma_plan_t* plan) {
    soma_opt* o = live_handle(h);
    if (!o) return SOMA_ERR_STATE;
    if (!plan) return o->fail(SOMA_ERR_INVALID_ARG, "plan is NULL");
    *plan = o->plan;
    return SOMA_OK;
}

soma_status_t soma_opt_get_segments(soma_opt_t h, int32_t which, soma_segment_t* out, int64_t cap,
                                    int64_t* count) {
    soma_opt* o = live_handle(h);
    if (!o) return SOMA_ERR_STATE;
    if (which != 0 && which != 1) return o->fail(SOMA_ERR_INVALID_ARG, "which must be 0 (update) or 1 (norm)");
    if (!count || cap < 0 || (cap > 0 && !out)) return o->fail(SOMA_ERR_INVALID_ARG, "bad output arguments");
    if (o->active < 0) return o->fail(SOMA_ERR_STATE, "no step has run on this handle yet");
    const soma::Table& t = which == 0 ? o->upd_tab : o->norm_tab;
    DeviceGuard dg(o->device);
    if (dg.status != cudaSuccess) return o->cuda_fail(dg.status, "cudaSetDevice");
    soma_status_t st = wait_idle(o);  // the tables' upload is ordered before the last step
    if (st != SOMA_OK) return st;
    std::vector<int32_t> begin((size_t)t.nchunks + 1);
    cudaError_t e = cudaMemcpy(begin.data(), t.chunk_begin, begin.size() * sizeof(int32_t), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return o->cuda_fail(e, "cudaMemcpy(chunk table)");
    const int64_t nseg = begin.back();
    *count = nseg;
    const int64_t take = std::min<int64_t>(cap, nseg);
    if (take == 0) return SOMA_OK;
    std::vector<soma::Seg> segs((size_t)take);
    if ((e = cudaMemcpy(segs.data(), t.segs, segs.size() * sizeof(soma::Seg), cudaMemcpyDeviceToHost)) != cudaSuccess)
        return o->cuda_fail(e, "cudaMemcpy(segment table)");
    int64_t c = 0;
    for (int64_t i = 0; i < take; ++i) {
        while (c + 1 < (int64_t)begin.size() && begin[(size_t)c + 1] <= i) ++c;
        const soma::Seg& sg = segs[(size_t)i];
        out[i] = soma_segment_t{sg.g, c, sg.len, sg.head, sg.nvec, (int32_t)sg.group};
    }
    return SOMA_OK;
}

soma_status_t soma_opt_get_cache_stats(soma_opt_t h, int64_t* builds, int64_t* reuses, int32_t* entries) {
    soma_opt* o = live_handle(h);
    if (!o) return SOMA_ERR_STATE;
    if (builds) *builds = o->plan_builds;
    if (reuses) *reuses = o->plan_reuses;
    if (entries) {
        int32_t k = 0;
        for (const auto& pl : o->plans) k += pl.valid ? 1 : 0;
        *entries = k;
    }
    return SOMA_OK;
}

void soma_opt_destroy(soma_opt_t h) {
    soma_opt* o = live_handle(h);
    if (!o) return;
    {
        std::lock_guard<std::mutex> lk(g_live_mu);
        g_live.erase(o);
    }
    if (o->dev_ready) {
        DeviceGuard dg(o->device);
        if (o->have_done) cudaEventSynchronize(o->done);
        if (o->groups_copy_pending) cudaEventSynchronize(o->groups_copied);
        for (auto& t3 : o->tev)
            for (auto& x : t3) cudaEventDestroy(x);
        if (o->done) cudaEventDestroy(o->done);
        if (o->d_res) cudaFree(o->d_res);
        if (o->d_partials) cudaFree(o->d_partials);
        for (auto& pl : o->plans)
            if (pl.d_tables) cudaFree(pl.d_tables);
        if (o->d_groups) cudaFree(o->d_groups);
        if (o->d_hp) cudaFree(o->d_hp);
        if (o->d_gscale) cudaFree(o->d_gscale);
        if (o->h_res) cudaFreeHost(o->h_res);
        if (o->h_staging) cudaFreeHost(o->h_staging);
        if (o->h_groups) cudaFreeHost(o->h_groups);
        if (o->groups_copied) cudaEventDestroy(o->groups_copied);
    }
    delete o;
}

}  // extern "C"
