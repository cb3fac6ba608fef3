// per_api.cu -- the C ABI of libgbper: argument checks, allocation, launches.  Every compute
// step runs in the kernels of k_tree.cu, k_sample.cu and k_rank.cu; this file only validates,
// allocates once at creation and enqueues work on the caller's stream.
#include "gbper.h"
#include "per_internal.cuh"

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <string>

using namespace gbper;

struct per_buffer {
    int device = 0;
    int num_sms = 1;
    uint64_t capacity = 0, n = 1;
    int D = 0;
    uint32_t d = 0, dp = 0;
    double alpha = 0.6, eps = 1e-6;
    uint32_t mode = PER_MODE_PROPORTIONAL;
    uint64_t seed = 0;
    // proportional
    float *L = nullptr;
    double *S = nullptr;
    float *M = nullptr;
    // rank
    RankWork rank{};
    // flat
    FlatWork flat{};
    void *flat_mem = nullptr;
    uint64_t flat_bytes = 0;
    // ring
    float *states = nullptr, *next = nullptr;
    uint32_t *actions = nullptr;
    float *rewards = nullptr;
    uint8_t *dones = nullptr;
    Ctl *ctl = nullptr;
    uint64_t host_size = 0, host_cursor = 0;
    // rank mode: the order kept between samples (keys/vals[merge_ctl[4]], order_size entries) and
    // an upper bound on the slots written since (each insertion or update adds its count)
    bool order_valid = false, always_resort = false;
    bool dones_f32 = false;   // per_sample writes dones as float
    // large-batch update: one winner word per slot (zero between calls) and the batch size from
    // which it is used (0: the measured default; UINT32_MAX: never)
    unsigned *win = nullptr;
    uint32_t rebuild_batch = 0;
    uint32_t element_batch = 0;   // per_config.element_batch
    // crowding of update batches (proportional mode): a host-mapped word the update kernels
    // write (crowd_host on the host, crowd_dev on the device) and the rebuild's subtree counts
    unsigned *crowd_host = nullptr, *crowd_dev = nullptr, *crowd_hist = nullptr;
    unsigned crowd_seen = 0xffffffffu;   // the last report acted on
    int upd_extra = 0;                   // the climb splits 2^upd_extra times as finely as by size
    bool upd_rebuild = false;            // crowding chose the rebuild
    uint64_t order_size = 0, dirty_bound = 0;
    unsigned *dirty_words = nullptr;   // slot marks [dirty_nwords] + list, old keys [kMaxDirty each] + control [8]
    uint64_t dirty_nwords = 0;         // words of slot marks (one per slot)
    std::string err;
};

namespace {

thread_local std::string g_create_err;

per_status fail(per_buffer *h, per_status s, const std::string &msg)
{
    if (h) h->err = msg;
    else g_create_err = msg;
    return s;
}

per_status cuda_fail(per_buffer *h, cudaError_t e, const char *where)
{
    return fail(h, PER_ERR_CUDA, std::string(where) + ": " + cudaGetErrorString(e));
}

TreeRefs tree_of(const per_buffer *h)
{
    TreeRefs t;
    t.L = h->L;
    t.S = h->S;
    t.M = h->M;
    t.n = h->n;
    t.D = h->D;
    return t;
}

RingRefs ring_of(const per_buffer *h)
{
    RingRefs r;
    r.states = h->states;
    r.next = h->next;
    r.actions = h->actions;
    r.rewards = h->rewards;
    r.dones = h->dones;
    r.capacity = h->capacity;
    r.d = h->d;
    return r;
}

void free_all(per_buffer *h)
{
    if (h->crowd_host) cudaFreeHost(h->crowd_host);
    void *ptrs[] = {h->L, h->S, h->M, h->rank.raw, h->rank.cdf, h->rank.guide, h->rank.keys[0], h->rank.keys[1],
                    h->rank.vals[0], h->rank.vals[1], h->rank.status, h->rank.digit_hist,
                    h->dirty_words, h->win, h->flat_mem, h->crowd_hist,
                    h->states, h->next, h->actions, h->rewards, h->dones, h->ctl};
    for (void *p : ptrs)
        if (p) cudaFree(p);
}

template <typename T>
bool alloc(T **p, uint64_t count)
{
    if (count == 0) count = 1;
    return cudaMalloc(reinterpret_cast<void **>(p), count * sizeof(T)) == cudaSuccess;
}

cudaStream_t as_stream(void *s) { return reinterpret_cast<cudaStream_t>(s); }

// Measured on GB300 (L2 flushed before each call): one entry propagates in about 10 us (the
// climb takes 16-21 us at any small batch), each further entry adds about 3 us, so one or two
// entries go entry by entry.
constexpr uint64_t kDefaultElementBatch = 3;

// The batch size from which per_update_priorities scatters (and, proportional, rebuilds every
// tree level) instead of climbing from each changed leaf: per_config.rebuild_batch, else the
// crossover measured on GB300 (L2 flushed before each call).  The rebuild costs about
// 16 us + 5 ns per leaf; the climb about 18-25 us up to a few thousand entries, then grows with
// the entries per subtree.  They meet near n/128 entries (2^21 leaves: 16384; 2^24: 131072);
// below 1024 entries the two are within the timer's 2 us resolution at every tree size.  In
// rank mode (no tree) the scatter is at least as fast as the climb at every batch size.
uint64_t update_rebuild_batch(const per_buffer *h)
{
    if (h->rebuild_batch == UINT32_MAX) return UINT64_MAX;
    if (h->rebuild_batch) return h->rebuild_batch;
    if (h->mode == PER_MODE_RANK) return 1;
    return std::max<uint64_t>(h->n / 128, 1024);
}

// Crowding.  The climb serves a subtree's entries 32 distinct leaves at a time, one group after
// the other, so a batch whose draws crowd a few subtrees (new rows entering at the running
// maximum keep most of the mass, say) climbs for several times as long.  The update kernels report
// the most entries one subtree received, with the split they used, through a word in mapped host
// memory (no synchronisation: it lags the enqueued calls by the few the GPU has not run yet).
// On each new report of the current split: above 32 entries, the next climbs split the tree twice
// as finely (up to 2^10 subtrees), which spreads a crowded stretch of slots over more warps; at
// most 8, once as coarsely again (down to the split for the batch size); and when even the finest
// split leaves at least 32 max(2, 5/6 leaves / 2^20) entries in a subtree (as many groups of 32
// as a rebuild's time buys), the next calls rebuild every level (the rebuild does not care where
// the entries fall) until its own subtree counts fall below that.  Measured on GB300 at 2^21 leaves, B = 512: 63 entries in one of 64 subtrees climbed in
// 22.6 us, as long as a rebuild, and lasting crowding of up to 465 climbed in 68-104 us against
// 33 us rebuilding.  per_config.rebuild_batch other than 0 keeps the size rule alone.  A call
// captured in a CUDA graph keeps the plan made at capture.  Returns the subtree count's log2 for
// the climb, or -1 for the rebuild.
int update_plan(per_buffer *h, unsigned B)
{
    const int base = update_subtree_log(B, h->D);
    const int pmax = std::min(kMaxUpdateLog, std::max(h->D - 1, 0));
    if (!h->crowd_host || h->rebuild_batch != 0) return base;
    const unsigned w = *reinterpret_cast<volatile const unsigned *>(h->crowd_host);
    if (w != h->crowd_seen) {
        h->crowd_seen = w;
        const int pm = (int)(w >> 28);   // the report's split; bits 20..27 a sequence number
        const uint64_t cnt = w & 0xfffffu;
        // a rebuild costs about 14 us + 4 ns a leaf, each further group of 32 leaves of a climb
        // about 5 us (measured on GB300): rebuild once a subtree needs more groups than that
        const uint64_t rebuild_at = 32 * std::max<uint64_t>(2, (h->n >> 20) * 5 / 6);
        const int cur = h->upd_rebuild ? pmax : std::min(base + h->upd_extra, pmax);
        if (w != 0 && pm == cur) {   // a report of the current plan
            if (h->upd_rebuild) {
                if (cnt < rebuild_at) h->upd_rebuild = false;
            } else if (cnt > 32) {
                if (cur < pmax) h->upd_extra = cur + 1 - base;
                else if (cnt >= rebuild_at) h->upd_rebuild = true;
            } else if (cnt <= 8 && h->upd_extra > 0) {
                h->upd_extra -= 1;
            }
        }
    }
    if (h->upd_rebuild) return -1;
    return std::min(base + std::max(h->upd_extra, 0), pmax);
}

// Proportional batches of fewer entries than this propagate entry by entry (per_config.element_batch,
// else the crossover measured on GB300).
uint64_t update_element_batch(const per_buffer *h)
{
    if (h->mode != PER_MODE_PROPORTIONAL || h->D == 0) return 0;
    if (h->element_batch) return h->element_batch;
    return kDefaultElementBatch;
}

// Rank mode: bring the slot order (keys/vals[merge_ctl[4]]) up to date for the filled slots.  When
// the order exists and at most kMaxDirty slots (and no more than an eighth of them) were written
// since, the written slots are merged into it; otherwise every slot is sorted again and the
// marks are cleared.  The decision uses host-side counts only (no synchronisation).
cudaError_t rank_order(per_buffer *h, cudaStream_t st)
{
    RankWork &w = h->rank;
    cudaError_t e;
    // nothing written since the order was made (per_rank_refresh just ran, say): it is current,
    // and sorting it again (PER_FLAG_RANK_RESORT) would give the same order
    if (h->order_valid && h->dirty_bound == 0 && h->order_size == h->host_size) return cudaSuccess;
    if (!h->always_resort && h->order_valid && h->dirty_bound <= kMaxDirty && h->dirty_bound * 8 <= h->host_size) {
        if (h->dirty_bound > 0) {
            e = launch_rank_merge(w, h->order_size, st);
            if (e != cudaSuccess) return e;
        }
    } else {
        // the sort's first kernel also opens a new mark epoch with an empty list
        unsigned *sorted = nullptr, *keys = nullptr;
        e = launch_rank_sort(w, h->host_size, &sorted, st, &keys);
        if (e != cudaSuccess) return e;
    }
    h->order_valid = true;
    h->order_size = h->host_size;
    h->dirty_bound = 0;
    return cudaSuccess;
}

// Kernel attributes are per device: set them the first time a buffer is created on a device.
// The carveout (percent of the unified L1/shared array preferred for shared memory; a kernel
// still gets the shared memory it needs), measured on GB300: the tree kernels but the level
// rebuild prefer L1 (0): the apex step 37.2K steps/s against 36.8K with the driver's choice
// (the rebuild's shared memory needs the larger configurations for more than one CTA per SM);
// the samplers keep the driver's choice (with 0 the stress sample took 35.6 us against 27.1);
// so do the rank kernels, which stage whole tiles in shared memory (-1: the driver's).
cudaError_t init_kernels_once(int device)
{
    static std::mutex mu;
    static bool done[64] = {};
    std::lock_guard<std::mutex> lock(mu);
    if (device < 0 || device >= 64) return cudaErrorInvalidDevice;
    if (done[device]) return cudaSuccess;
    const int tree_carveout = 0, sample_carveout = -1, rank_carveout = -1;
    cudaError_t e = init_tree_kernels(tree_carveout);
    if (e == cudaSuccess) e = init_sample_kernels(sample_carveout);
    if (e == cudaSuccess) e = init_rank_kernels(rank_carveout);
    if (e == cudaSuccess) done[device] = true;
    return e;
}

}  // namespace

namespace gbper {
// Programmatic dependent launch for every hot kernel (measured on GB300: 0.7-0.8 us between
// consecutive kernels against 3-4.5 us without it).
bool pdl_enabled() { return true; }
}  // namespace gbper

extern "C" {

per_status per_create(uint64_t capacity, uint32_t state_dim, const per_config *cfg, per_buffer **out)
{
    g_create_err.clear();
    if (!out) return fail(nullptr, PER_ERR_INVALID_ARG, "per_create: out is NULL");
    if (capacity == 0 || capacity > (1ull << 31))
        return fail(nullptr, PER_ERR_INVALID_ARG, "per_create: capacity must be in 1 .. 2^31");
    if (state_dim > 65536) return fail(nullptr, PER_ERR_INVALID_ARG, "per_create: state_dim > 65536");
    per_config c;
    if (cfg) {
        c = *cfg;
    } else {
        std::memset(&c, 0, sizeof(c));
        c.alpha = 0.6;
        c.eps = 1e-6;
    }
    if (c.row_stride_out == 0) c.row_stride_out = state_dim;
    if (c.row_stride_out < state_dim)
        return fail(nullptr, PER_ERR_INVALID_ARG, "per_create: row_stride_out < state_dim");
    if (c.row_stride_out > 65536) return fail(nullptr, PER_ERR_INVALID_ARG, "per_create: row_stride_out > 65536");
    if (!(c.alpha >= 0.0) || !std::isfinite(c.alpha))
        return fail(nullptr, PER_ERR_INVALID_ARG, "per_create: alpha must be finite and >= 0");
    if (!(c.eps > 0.0) || !std::isfinite(c.eps))
        return fail(nullptr, PER_ERR_INVALID_ARG, "per_create: eps must be finite and > 0");
    if (c.mode != PER_MODE_PROPORTIONAL && c.mode != PER_MODE_RANK && c.mode != PER_MODE_UNIFORM &&
        c.mode != PER_MODE_FLAT)
        return fail(nullptr, PER_ERR_INVALID_ARG, "per_create: unknown mode");
    if (c.reserved != 0) return fail(nullptr, PER_ERR_INVALID_ARG, "per_create: reserved must be 0");
    if (c.flags & ~(PER_FLAG_RANK_RESORT | PER_FLAG_DONES_F32))
        return fail(nullptr, PER_ERR_INVALID_ARG, "per_create: unknown flags");
    if (c.mode == PER_MODE_FLAT && c.alpha > 1.0)
        return fail(nullptr, PER_ERR_INVALID_ARG,
                    "per_create: flat mode needs alpha <= 1 (every leaf then stays a finite binary32)");
    if ((c.mode == PER_MODE_PROPORTIONAL || c.mode == PER_MODE_FLAT) &&
        !((float)std::pow(c.eps, c.alpha) >= 1.17549435e-38f))
        return fail(nullptr, PER_ERR_INVALID_ARG,
                    "per_create: eps^alpha underflows binary32; a leaf of 0 would read as an empty slot");

    per_buffer *h = new (std::nothrow) per_buffer();
    if (!h) return fail(nullptr, PER_ERR_OOM, "per_create: host allocation failed");
    cudaError_t e = cudaGetDevice(&h->device);
    if (e != cudaSuccess) {
        delete h;
        return fail(nullptr, PER_ERR_CUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(e));
    }
    cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, h->device);
    e = init_kernels_once(h->device);
    if (e != cudaSuccess) {
        delete h;
        return fail(nullptr, PER_ERR_CUDA, std::string("kernel attributes: ") + cudaGetErrorString(e));
    }
    if (h->num_sms < 1) h->num_sms = 1;
    h->capacity = capacity;
    while (h->n < capacity) {
        h->n <<= 1;
        h->D += 1;
    }
    h->d = state_dim;
    h->dp = c.row_stride_out;
    h->alpha = c.alpha;
    h->eps = c.eps;
    h->mode = c.mode;
    h->seed = c.seed;
    h->always_resort = (c.flags & PER_FLAG_RANK_RESORT) != 0;
    h->dones_f32 = (c.flags & PER_FLAG_DONES_F32) != 0;
    h->rebuild_batch = c.rebuild_batch;
    h->element_batch = c.element_batch;

    bool ok = alloc(&h->ctl, 1);
    if (c.mode == PER_MODE_PROPORTIONAL) {
        ok = ok && alloc(&h->L, h->n) && alloc(&h->S, h->n) && alloc(&h->M, h->n) && alloc(&h->win, h->n) &&
             alloc(&h->crowd_hist, 1024);
        if (ok && h->D > 0) {
            void *hp = nullptr, *dp = nullptr;
            ok = cudaHostAlloc(&hp, 64, cudaHostAllocMapped) == cudaSuccess;
            if (ok) {
                h->crowd_host = static_cast<unsigned *>(hp);
                std::memset(hp, 0, 64);
                ok = cudaHostGetDevicePointer(&dp, hp, 0) == cudaSuccess;
                h->crowd_dev = static_cast<unsigned *>(dp);
            }
        }
    } else if (c.mode == PER_MODE_FLAT) {
        // one block: C [capacity] f64, tile sums and offsets (u64 each), the result words, tile
        // minima f32, tickets
        const uint64_t tiles = flat_tiles(capacity);
        const uint64_t bytes = 8 * capacity + tiles * (8 + 16 + 4) + 4 * 8 + 2 * 4;
        ok = ok && alloc(&h->L, h->n) && alloc(&h->win, capacity) &&
             cudaMalloc(&h->flat_mem, bytes) == cudaSuccess;
        if (ok) {
            char *p = static_cast<char *>(h->flat_mem);
            h->flat.C = reinterpret_cast<double *>(p);
            p += 8 * capacity;
            h->flat.agg = reinterpret_cast<unsigned long long *>(p);
            p += 8 * tiles;
            h->flat.excl = reinterpret_cast<unsigned long long *>(p);
            p += 16 * tiles;
            h->flat.res = reinterpret_cast<unsigned long long *>(p);
            p += 4 * 8;
            h->flat.tmin = reinterpret_cast<float *>(p);
            p += 4 * tiles;
            h->flat.tick = reinterpret_cast<unsigned *>(p);
            h->flat_bytes = bytes;
        }
    } else if (c.mode == PER_MODE_RANK) {
        ok = ok && alloc(&h->rank.raw, capacity) && alloc(&h->rank.cdf, capacity + 1) &&
             alloc(&h->rank.keys[0], capacity) && alloc(&h->rank.keys[1], capacity) &&
             alloc(&h->rank.vals[0], capacity) && alloc(&h->rank.vals[1], capacity) &&
             alloc(&h->rank.status, rank_status_words(capacity)) && alloc(&h->rank.digit_hist, 4 * 256 + 16) &&
             alloc(&h->win, capacity);
        h->rank.sort_ctl = h->rank.digit_hist + 4 * 256;
        h->rank.capacity = capacity;
        h->rank.num_sms = h->num_sms;
        h->dirty_nwords = capacity;   // one mark epoch per slot
        ok = ok && alloc(&h->dirty_words, h->dirty_nwords + 2 * kMaxDirty + 8);
        if (ok) {
            h->rank.dirty.mark = h->dirty_words;
            h->rank.dirty.list = h->dirty_words + h->dirty_nwords;
            h->rank.dirty.oldkey = h->rank.dirty.list + kMaxDirty;
            // [1] mark epoch, [2] merge arrivals, [3] listed count, [4] which pair holds the order
            h->rank.merge_ctl = h->rank.dirty.oldkey + kMaxDirty;
            h->rank.dirty.epoch = h->rank.merge_ctl + 1;
            h->rank.dirty.count = h->rank.merge_ctl + 3;
        }
    }
    ok = ok && alloc(&h->states, capacity * (uint64_t)state_dim) && alloc(&h->next, capacity * (uint64_t)state_dim) &&
         alloc(&h->actions, capacity) && alloc(&h->rewards, capacity) && alloc(&h->dones, capacity);
    if (!ok) {
        cudaGetLastError();
        free_all(h);
        delete h;
        return fail(nullptr, PER_ERR_OOM, "per_create: device allocation failed");
    }
    Ctl init;
    std::memset(&init, 0, sizeof(init));
    const float one = 1.0f;
    std::memcpy(&init.max_raw_bits, &one, sizeof(one));
    std::memcpy(&init.max_leaf_bits, &one, sizeof(one));  // pow(1, alpha) = 1
    e = cudaMemcpy(h->ctl, &init, sizeof(init), cudaMemcpyHostToDevice);
    if (e == cudaSuccess && h->L) e = cudaMemset(h->L, 0, h->n * sizeof(float));
    if (e == cudaSuccess && h->S) e = cudaMemset(h->S, 0, h->n * sizeof(double));
    if (e == cudaSuccess && h->M) e = launch_fill_mins(h->M, h->n, 0);
    if (e == cudaSuccess && h->rank.raw) e = cudaMemset(h->rank.raw, 0, capacity * sizeof(float));
    if (e == cudaSuccess && h->win) e = cudaMemset(h->win, 0, (h->S ? h->n : capacity) * sizeof(unsigned));
    if (e == cudaSuccess && h->crowd_hist) e = cudaMemset(h->crowd_hist, 0, 1024 * sizeof(unsigned));
    if (e == cudaSuccess && h->flat_mem) e = cudaMemset(h->flat_mem, 0, h->flat_bytes);
    if (e == cudaSuccess && h->rank.status)
        e = cudaMemset(h->rank.status, 0, rank_status_words(capacity) * sizeof(unsigned long long));
    if (e == cudaSuccess && h->rank.digit_hist) e = cudaMemset(h->rank.digit_hist, 0, (4 * 256 + 16) * sizeof(unsigned));
    if (e == cudaSuccess && h->dirty_words)
        e = cudaMemset(h->dirty_words, 0, (h->dirty_nwords + 2 * kMaxDirty + 8) * sizeof(unsigned));
    if (e == cudaSuccess && h->dirty_words) {   // the first mark epoch is 1: no slot is marked
        const unsigned one_epoch = 1u;
        e = cudaMemcpy(h->rank.merge_ctl + 1, &one_epoch, sizeof(one_epoch), cudaMemcpyHostToDevice);
    }
    if (h->rank.raw) h->rank.err = &h->ctl->err_flags;
    if (e == cudaSuccess && h->rank.cdf) e = launch_build_cdf(h->rank.cdf, capacity, h->alpha, 0);
    if (e == cudaSuccess && h->rank.cdf) {
        // the CDF's guide: buckets of mass at most two ranks' mass where ranks are sparsest in
        // mass (the last, each of mass capacity^-alpha), so that each bucket holds at most three
        // candidate ranks, with at most two buckets per slot (beyond that, the sparsest buckets
        // hold more and the sampler searches them).  The bucket width delta is a power of two, so
        // k delta is exact and a mass's bucket is the truncation of one exact product.
        double T = 0.0;
        e = cudaMemcpy(&T, h->rank.cdf + capacity, sizeof(double), cudaMemcpyDeviceToHost);
        uint64_t cap2 = 2;
        while (cap2 < capacity) cap2 <<= 1;
        cap2 *= 2;
        const double dmax = 2.0 / std::pow((double)capacity, h->alpha);   // at most two ranks' mass
        double delta = std::ldexp(1.0, (int)std::floor(std::log2(dmax)));   // the largest power of two <= dmax
        while (delta * 2.0 <= dmax) delta *= 2.0;
        while (delta > dmax) delta *= 0.5;
        while (std::ceil(T / delta) > (double)cap2) delta *= 2.0;
        const uint64_t K = std::max<uint64_t>((uint64_t)std::ceil(T / delta), 1);
        if (e == cudaSuccess && !alloc(&h->rank.guide, K + 1)) {
            cudaGetLastError();
            free_all(h);
            delete h;
            return fail(nullptr, PER_ERR_OOM, "per_create: device allocation failed");
        }
        h->rank.guide_k = (unsigned)K;
        h->rank.guide_delta = delta;
        if (e == cudaSuccess) e = launch_build_guide(h->rank.cdf, capacity, h->rank.guide, (unsigned)K,
                                                     h->rank.guide_delta, 0);
    }
    if (e == cudaSuccess && state_dim) e = cudaMemset(h->states, 0, capacity * (uint64_t)state_dim * sizeof(float));
    if (e == cudaSuccess && state_dim) e = cudaMemset(h->next, 0, capacity * (uint64_t)state_dim * sizeof(float));
    if (e == cudaSuccess) e = cudaMemset(h->actions, 0, capacity * sizeof(uint32_t));
    if (e == cudaSuccess) e = cudaMemset(h->rewards, 0, capacity * sizeof(float));
    if (e == cudaSuccess) e = cudaMemset(h->dones, 0, capacity);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
        free_all(h);
        delete h;
        return fail(nullptr, PER_ERR_CUDA, std::string("per_create init: ") + cudaGetErrorString(e));
    }
    *out = h;
    return PER_OK;
}

per_status per_destroy(per_buffer *h)
{
    if (!h) return PER_OK;
    int cur = 0;
    cudaGetDevice(&cur);
    if (cur != h->device) cudaSetDevice(h->device);
    cudaDeviceSynchronize();
    free_all(h);
    if (cur != h->device) cudaSetDevice(cur);
    delete h;
    return PER_OK;
}

per_status per_add(per_buffer *h, uint64_t count, const float *d_states, const float *d_next,
                   const uint32_t *d_actions, const float *d_rewards, const uint8_t *d_dones,
                   const float *d_raw_prio, void *stream)
{
    if (!h) return PER_ERR_INVALID_ARG;
    if (count == 0) return PER_OK;
    if (!d_actions || !d_rewards || !d_dones)
        return fail(h, PER_ERR_INVALID_ARG, "per_add: actions, rewards and dones are required");
    if (h->d && (!d_states || !d_next))
        return fail(h, PER_ERR_INVALID_ARG, "per_add: states and next_states are required");
    if (h->d && ((reinterpret_cast<uintptr_t>(d_states) | reinterpret_cast<uintptr_t>(d_next)) % 4))
        return fail(h, PER_ERR_INVALID_ARG, "per_add: row arrays must be 4-byte aligned");
    if ((reinterpret_cast<uintptr_t>(d_actions) | reinterpret_cast<uintptr_t>(d_rewards)) % 4 ||
        (d_raw_prio && reinterpret_cast<uintptr_t>(d_raw_prio) % 4))
        return fail(h, PER_ERR_INVALID_ARG, "per_add: scalar arrays must be 4-byte aligned");
    if (count > (1ull << 40)) return fail(h, PER_ERR_INVALID_ARG, "per_add: count too large");
    bool marked = false;
    const cudaError_t e = launch_add(tree_of(h), ring_of(h), h->rank.raw, h->ctl, count, d_states, d_next,
                                     d_actions, d_rewards, d_dones, d_raw_prio, h->alpha, h->eps,
                                     h->mode == PER_MODE_PROPORTIONAL || h->mode == PER_MODE_FLAT,
                                     h->host_cursor, h->num_sms,
                                     h->rank.dirty, h->mode == PER_MODE_RANK ? h->rank.cdf : nullptr, &marked,
                                     as_stream(stream));
    if (e != cudaSuccess) return cuda_fail(h, e, "per_add launch");
    if (h->mode == PER_MODE_RANK) {
        if (marked) h->dirty_bound += count;
        else h->order_valid = false;   // rewritten in bulk, unmarked: the next sample sorts again
    }
    h->host_cursor = (h->host_cursor + count) % h->capacity;
    h->host_size = std::min<uint64_t>(h->host_size + count, h->capacity);
    return PER_OK;
}

per_status per_sample(per_buffer *h, uint32_t B, float beta, int64_t *d_idx, float *d_w, float *d_states,
                      float *d_next, uint32_t *d_actions, float *d_rewards, uint8_t *d_dones, void *stream)
{
    if (!h) return PER_ERR_INVALID_ARG;
    if (B == 0 || B > (1u << 24)) return fail(h, PER_ERR_INVALID_ARG, "per_sample: B must be in 1 .. 2^24");
    if (!d_idx) return fail(h, PER_ERR_INVALID_ARG, "per_sample: d_idx is required");
    if (!(beta >= 0.0f) || !std::isfinite(beta))
        return fail(h, PER_ERR_INVALID_ARG, "per_sample: beta must be finite and >= 0");
    if (reinterpret_cast<uintptr_t>(d_idx) % 8 || reinterpret_cast<uintptr_t>(d_w) % 4 ||
        reinterpret_cast<uintptr_t>(d_states) % 4 || reinterpret_cast<uintptr_t>(d_next) % 4 ||
        reinterpret_cast<uintptr_t>(d_actions) % 4 || reinterpret_cast<uintptr_t>(d_rewards) % 4 ||
        (h->dones_f32 && reinterpret_cast<uintptr_t>(d_dones) % 4))
        return fail(h, PER_ERR_INVALID_ARG, "per_sample: misaligned output pointer");
    if (h->host_size == 0) return fail(h, PER_ERR_EMPTY, "per_sample: the buffer holds no transition");
    if (h->mode == PER_MODE_RANK && h->host_size < h->capacity) {
        // the slot order's length is a launch argument: a graph captured now would keep sorting
        // this many slots while later replays fill the buffer further
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(as_stream(stream), &cs) == cudaSuccess && cs != cudaStreamCaptureStatusNone)
            return fail(h, PER_ERR_INVALID_ARG,
                        "per_sample: in rank mode, capture a graph only once the buffer is full");
    }
    SampleOut o;
    o.idx = reinterpret_cast<long long *>(d_idx);
    o.w = d_w;
    o.states = d_states;
    o.next = d_next;
    o.actions = d_actions;
    o.rewards = d_rewards;
    o.dones = d_dones;
    o.dones_f32 = h->dones_f32 ? 1 : 0;
    o.dp = h->dp;
    cudaError_t e;
    if (h->mode == PER_MODE_PROPORTIONAL) {
        e = launch_sample_prop(tree_of(h), ring_of(h), h->ctl, B, beta, h->seed, o, h->num_sms, as_stream(stream));
    } else if (h->mode == PER_MODE_UNIFORM) {
        e = launch_sample_uniform(ring_of(h), h->ctl, B, h->seed, o, h->num_sms, as_stream(stream));
    } else if (h->mode == PER_MODE_FLAT) {
        e = launch_flat_scan(h->L, h->flat, h->ctl, h->capacity, as_stream(stream));
        if (e == cudaSuccess)
            e = launch_sample_flat(h->L, h->flat, ring_of(h), h->ctl, B, beta, h->seed, o, h->num_sms,
                                   as_stream(stream));
    } else {
        e = rank_order(h, as_stream(stream));
        const unsigned *sorted = h->rank.vals[1];   // unused: the kernel reads the order's buffer
        if (e == cudaSuccess)
            e = launch_sample_rank(h->rank, sorted, ring_of(h), h->ctl, B, beta, h->alpha, h->seed, o,
                                   h->num_sms, as_stream(stream));
    }
    if (e != cudaSuccess) return cuda_fail(h, e, "per_sample launch");
    return PER_OK;
}

per_status per_rank_refresh(per_buffer *h, void *stream)
{
    if (!h) return PER_ERR_INVALID_ARG;
    if (h->mode != PER_MODE_RANK) return fail(h, PER_ERR_INVALID_ARG, "per_rank_refresh: rank mode only");
    if (h->host_size == 0) return PER_OK;   // no filled slot: nothing to order
    if (h->host_size < h->capacity) {
        // as in per_sample: the order's length is a launch argument
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(as_stream(stream), &cs) == cudaSuccess && cs != cudaStreamCaptureStatusNone)
            return fail(h, PER_ERR_INVALID_ARG,
                        "per_rank_refresh: capture a graph only once the buffer is full");
    }
    const cudaError_t e = rank_order(h, as_stream(stream));
    return e == cudaSuccess ? PER_OK : cuda_fail(h, e, "per_rank_refresh launch");
}

per_status per_update_priorities(per_buffer *h, uint32_t B, const int64_t *d_idx, const float *d_td,
                                 void *stream)
{
    if (!h) return PER_ERR_INVALID_ARG;
    if (B == 0) return PER_OK;
    if (B > (1u << 24)) return fail(h, PER_ERR_INVALID_ARG, "per_update_priorities: B > 2^24");
    if (!d_idx || !d_td) return fail(h, PER_ERR_INVALID_ARG, "per_update_priorities: NULL input");
    if (reinterpret_cast<uintptr_t>(d_idx) % 8 || reinterpret_cast<uintptr_t>(d_td) % 4)
        return fail(h, PER_ERR_INVALID_ARG, "per_update_priorities: misaligned input");
    if (h->mode == PER_MODE_UNIFORM) return PER_OK;   // no priorities
    const long long *idx = reinterpret_cast<const long long *>(d_idx);
    const bool prop = h->mode == PER_MODE_PROPORTIONAL || h->mode == PER_MODE_FLAT;
    cudaStream_t st = as_stream(stream);
    cudaError_t e;
    const CrowdRefs none{nullptr, nullptr, 0, 0};
    if (B < update_element_batch(h)) {
        // one or two entries: each from its leaf to the root
        e = launch_update_element(tree_of(h), h->ctl, B, idx, d_td, h->alpha, h->eps, st);
    } else if (h->mode == PER_MODE_FLAT || B >= update_rebuild_batch(h)) {
        // winners scattered, then (with a tree) every level rebuilt
        e = launch_update_rebuild(tree_of(h), h->rank.raw, h->ctl, B, idx, d_td, h->alpha, h->eps, prop,
                                  h->num_sms, h->rank.dirty, h->win, none, st);
    } else {
        const int P = h->mode == PER_MODE_PROPORTIONAL ? update_plan(h, B) : -1;
        if (h->mode == PER_MODE_PROPORTIONAL && P < 0) {
            // the rebuild, chosen because recent batches crowded even the finest split; the
            // crowding is measured on the way (at that split), so the choice can return
            const int pf = std::min(kMaxUpdateLog, std::max(h->D - 1, 0));
            const CrowdRefs c{h->crowd_dev, h->crowd_hist, h->D - pf, 1u << pf};
            e = launch_update_rebuild(tree_of(h), h->rank.raw, h->ctl, B, idx, d_td, h->alpha, h->eps, prop,
                                      h->num_sms, h->rank.dirty, h->win, c, st);
        } else {
            // the dirty-ancestor climb over 2^P subtrees (measuring the crowding)
            const CrowdRefs c{h->crowd_dev, nullptr, 0, 0};
            e = launch_update(tree_of(h), h->rank.raw, h->ctl, B, idx, d_td, h->alpha, h->eps, prop, h->num_sms,
                              h->rank.dirty, c, P, st);
        }
    }
    if (e != cudaSuccess) return cuda_fail(h, e, "per_update_priorities launch");
    if (h->mode == PER_MODE_RANK) h->dirty_bound += B;
    return PER_OK;
}

per_status per_total(per_buffer *h, double *host_out, void *stream)
{
    if (!h || !host_out) return PER_ERR_INVALID_ARG;
    cudaStream_t st = as_stream(stream);
    cudaError_t e;
    if (h->mode == PER_MODE_UNIFORM) {
        uint64_t size = 0;
        e = cudaMemcpyAsync(&size, &h->ctl->size, sizeof(size), cudaMemcpyDeviceToHost, st);
        if (e == cudaSuccess) e = cudaStreamSynchronize(st);
        *host_out = (double)size;
        return e == cudaSuccess ? PER_OK : cuda_fail(h, e, "per_total");
    } else if (h->mode == PER_MODE_FLAT) {
        if (h->host_size == 0) {
            *host_out = 0.0;
            return PER_OK;
        }
        e = launch_flat_scan(h->L, h->flat, h->ctl, h->capacity, st);
        if (e == cudaSuccess) e = cudaMemcpyAsync(host_out, h->flat.res + 1, sizeof(double), cudaMemcpyDeviceToHost, st);
    } else if (h->mode == PER_MODE_RANK) {
        e = cudaMemcpyAsync(host_out, h->rank.cdf + h->host_size, sizeof(double), cudaMemcpyDeviceToHost, st);
    } else if (h->D == 0) {
        float v = 0.0f;
        e = cudaMemcpyAsync(&v, h->L, sizeof(float), cudaMemcpyDeviceToHost, st);
        if (e == cudaSuccess) e = cudaStreamSynchronize(st);
        *host_out = (double)v;
        return e == cudaSuccess ? PER_OK : cuda_fail(h, e, "per_total");
    } else {
        e = cudaMemcpyAsync(host_out, h->S + 1, sizeof(double), cudaMemcpyDeviceToHost, st);
    }
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    return e == cudaSuccess ? PER_OK : cuda_fail(h, e, "per_total");
}

per_status per_min(per_buffer *h, float *host_out, void *stream)
{
    if (!h || !host_out) return PER_ERR_INVALID_ARG;
    if (h->mode != PER_MODE_PROPORTIONAL && h->mode != PER_MODE_FLAT)
        return fail(h, PER_ERR_INVALID_ARG, "per_min: proportional and flat modes only");
    if (h->host_size == 0) return fail(h, PER_ERR_EMPTY, "per_min: the buffer holds no transition");
    cudaStream_t st = as_stream(stream);
    cudaError_t e;
    float v = 0.0f;
    if (h->mode == PER_MODE_FLAT) {
        unsigned long long bits = 0;
        e = launch_flat_scan(h->L, h->flat, h->ctl, h->capacity, st);
        if (e == cudaSuccess) e = cudaMemcpyAsync(&bits, h->flat.res + 2, sizeof(bits), cudaMemcpyDeviceToHost, st);
        if (e == cudaSuccess) e = cudaStreamSynchronize(st);
        if (e != cudaSuccess) return cuda_fail(h, e, "per_min");
        const unsigned b32 = (unsigned)bits;
        std::memcpy(&v, &b32, sizeof(v));
        *host_out = v;
        return PER_OK;
    }
    if (h->D == 0) {
        e = cudaMemcpyAsync(&v, h->L, sizeof(float), cudaMemcpyDeviceToHost, st);
    } else {
        e = cudaMemcpyAsync(&v, h->M + 1, sizeof(float), cudaMemcpyDeviceToHost, st);
    }
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(h, e, "per_min");
    *host_out = v;
    return PER_OK;
}

per_status per_size(const per_buffer *h, uint64_t *out)
{
    if (!h || !out) return PER_ERR_INVALID_ARG;
    *out = h->host_size;
    return PER_OK;
}

per_status per_nleaves(const per_buffer *h, uint64_t *out)
{
    if (!h || !out) return PER_ERR_INVALID_ARG;
    *out = h->n;
    return PER_OK;
}

per_status per_status_device(per_buffer *h, uint32_t *host_flags, void *stream)
{
    if (!h) return PER_ERR_INVALID_ARG;
    cudaStream_t st = as_stream(stream);
    uint32_t flags = 0;
    cudaError_t e = cudaMemcpyAsync(&flags, &h->ctl->err_flags, sizeof(flags), cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(&h->ctl->err_flags, 0, sizeof(uint32_t), st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(h, e, "per_status_device");
    if (host_flags) *host_flags = flags;
    return flags ? PER_ERR_DEVICE_FLAG : PER_OK;
}

const char *per_last_error(const per_buffer *h)
{
    return h ? h->err.c_str() : g_create_err.c_str();
}

per_status per_read_state(per_buffer *h, uint32_t which, uint64_t first, uint64_t count, void *host_dst,
                          void *stream)
{
    if (!h || (!host_dst && count)) return PER_ERR_INVALID_ARG;
    const void *src = nullptr;
    uint64_t elems = 0, esz = 0;
    switch (which) {
    case PER_STATE_LEAVES: src = h->L; elems = h->n; esz = 4; break;
    case PER_STATE_SUMS: src = h->S; elems = h->n; esz = 8; break;
    case PER_STATE_MINS: src = h->M; elems = h->n; esz = 4; break;
    case PER_STATE_RAW: src = h->rank.raw; elems = h->capacity; esz = 4; break;
    case PER_STATE_CDF: src = h->rank.cdf; elems = h->capacity + 1; esz = 8; break;
    case PER_STATE_STATES: src = h->states; elems = h->capacity * (uint64_t)h->d; esz = 4; break;
    case PER_STATE_NEXT: src = h->next; elems = h->capacity * (uint64_t)h->d; esz = 4; break;
    case PER_STATE_ACTIONS: src = h->actions; elems = h->capacity; esz = 4; break;
    case PER_STATE_REWARDS: src = h->rewards; elems = h->capacity; esz = 4; break;
    case PER_STATE_DONES: src = h->dones; elems = h->capacity; esz = 1; break;
    case PER_STATE_RANK_ORDER:
        if (h->mode != PER_MODE_RANK || !h->order_valid)
            return fail(h, PER_ERR_INVALID_ARG, "per_read_state: no rank order yet (rank mode, after a sample)");
        {
            unsigned cur = 0;
            cudaError_t e = cudaMemcpyAsync(&cur, h->rank.merge_ctl + 4, sizeof(cur), cudaMemcpyDeviceToHost,
                                            as_stream(stream));
            if (e == cudaSuccess) e = cudaStreamSynchronize(as_stream(stream));
            if (e != cudaSuccess) return cuda_fail(h, e, "per_read_state");
            src = h->rank.vals[cur & 1u];
        }
        elems = h->order_size;
        esz = 4;
        break;
    case PER_STATE_CUMULATIVE: {
        if (h->mode != PER_MODE_FLAT) return fail(h, PER_ERR_INVALID_ARG, "per_read_state: flat mode only");
        // the device's filled size (graph replays advance it without the host counting)
        uint64_t dsize = 0;
        cudaError_t e = cudaMemcpyAsync(&dsize, &h->ctl->size, sizeof(dsize), cudaMemcpyDeviceToHost,
                                        as_stream(stream));
        if (e == cudaSuccess) e = cudaStreamSynchronize(as_stream(stream));
        if (e != cudaSuccess) return cuda_fail(h, e, "per_read_state");
        src = h->flat.C;
        elems = dsize;
        esz = 8;
        break;
    }
    case PER_STATE_COUNTERS: {
        if (first > 5 || count > 5 - first) return fail(h, PER_ERR_INVALID_ARG, "per_read_state: range");
        Ctl c;
        cudaStream_t st = as_stream(stream);
        cudaError_t e = cudaMemcpyAsync(&c, h->ctl, sizeof(Ctl), cudaMemcpyDeviceToHost, st);
        if (e == cudaSuccess) e = cudaStreamSynchronize(st);
        if (e != cudaSuccess) return cuda_fail(h, e, "per_read_state");
        const uint64_t crowd = h->crowd_host ? *reinterpret_cast<volatile const unsigned *>(h->crowd_host) : 0u;
        const uint64_t v[5] = {c.call_tix >> kCallShift, c.cursor, c.size, c.max_raw_bits, crowd};
        std::memcpy(host_dst, v + first, count * sizeof(uint64_t));
        return PER_OK;
    }
    default: return fail(h, PER_ERR_INVALID_ARG, "per_read_state: unknown array");
    }
    if (!src) return fail(h, PER_ERR_INVALID_ARG, "per_read_state: array absent in this mode");
    if (first > elems || count > elems - first) return fail(h, PER_ERR_INVALID_ARG, "per_read_state: range");
    if (count == 0) return PER_OK;
    cudaStream_t st = as_stream(stream);
    cudaError_t e = cudaMemcpyAsync(host_dst, static_cast<const char *>(src) + first * esz, count * esz,
                                    cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    return e == cudaSuccess ? PER_OK : cuda_fail(h, e, "per_read_state");
}

}  // extern "C"
