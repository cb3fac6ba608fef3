// per_internal.cuh -- shared declarations of the CUDA side of libgbper (sm_103a).
//
// Device layout of one replay buffer (proportional mode), n = 2^D leaves >= capacity:
//   L  float  [n]  leaves p^alpha; 0 marks an empty slot or a padding leaf
//   S  double [n]  internal sums, node i in [1, n): children 2i, 2i+1; nodes >= n are leaves
//   M  float  [n]  internal mins over filled leaves (+inf where none)
// Levels are contiguous: depth l holds nodes [2^l, 2^(l+1)), so a level is one coalesced
// stretch and every level from depth 4 down starts on a 128-byte line.
// Rank mode keeps raw priorities [capacity] and the rank CDF [capacity + 1] instead.
// The ring holds states / next_states [capacity x state_dim], actions, rewards, dones.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace gbper {

// Device-resident control block: counters that kernels advance themselves, so that a call
// replayed from a CUDA graph still draws a fresh batch and inserts at the right slot
// ("True Single-Graph Implementation Plan", Task 4: device-side counters).
struct Ctl {
    unsigned long long call_tix;      // sample calls << 24 | CTAs of the current call that started
    unsigned long long cursor;        // next ring slot
    unsigned long long size;          // filled slots
    unsigned int max_raw_bits;        // running maximum raw priority (float bits, > 0)
    unsigned int err_flags;           // PER_DEVFLAG_* bits
    unsigned int ticket_rebuild;      // arrivals in a full tree rebuild
    unsigned int ticket_update;
    unsigned int ticket_add;
    unsigned int batch_max_bits;      // per-call maximum raw priority, folded in by the last CTA
    unsigned int add_max_bits;
    unsigned int max_leaf_bits;       // fl32(pow(running maximum, alpha)): the leaf of a new row
    unsigned int crowd_max;           // the update's most entries in one subtree (reset by the top CTA)
    unsigned int crowd_seq;           // crowding reports made
    unsigned long long rank_total_bits;   // rank mode: cdf[size] (binary64 bits), kept with size
};

// A crowding report: (P << 28) | (sequence mod 256) << 20 | min(entries, 2^20 - 1).
__device__ __forceinline__ unsigned crowd_word(int P, unsigned seq, unsigned entries)
{
    return ((unsigned)P << 28) | ((seq & 0xffu) << 20) | min(entries, 0xfffffu);
}

__device__ __forceinline__ unsigned crowd_report(Ctl *c, int P, unsigned entries)
{
    return crowd_word(P, atomicAdd(&c->crowd_seq, 1u), entries);
}

// Crowding of update batches (proportional mode): the most entries one update subtree receives,
// written with the subtree count's log2 P and a sequence number (crowd_report) to host-mapped
// memory, for the
// host's choice of the update's subtrees and between climbing and rebuilding (see
// per_update_priorities).  The climb measures it while filing its batch; a rebuild chosen because
// of crowding measures it with a histogram of 2^P subtrees (P the climb's subtree count for the
// batch) so that the choice can return to the climb.
struct CrowdRefs {
    unsigned *host;    // device alias of the host-mapped word; null: not measured
    unsigned *hist;    // [1024] per-subtree counts (rebuild path), zero between calls; null: not kept
    int shift;         // slot >> shift is the subtree (rebuild path)
    unsigned nsub;     // subtrees (rebuild path)
};

// Fold a call's maximum raw priority into the running maximum and keep the cached leaf value
// of the maximum in step (one binary64 pow, only when the maximum rises).  Last CTA only.
__device__ __forceinline__ void fold_running_max(Ctl *c, unsigned call_max_bits, double alpha)
{
    if (call_max_bits > c->max_raw_bits) {
        c->max_raw_bits = call_max_bits;
        c->max_leaf_bits = __float_as_uint(__double2float_rn(pow((double)__uint_as_float(call_max_bits), alpha)));
    }
}

// The Philox call number of a sample launch, taken by each CTA at its start: one 64-bit atomic
// returns the call count (high 40 bits) and this CTA's arrival index (low 24 bits); the last CTA
// to arrive rolls the count over, so no CTA waits and none needs a fence at its end.
constexpr int kCallShift = 24;
__device__ __forceinline__ unsigned long long take_call_number(Ctl *c)
{
    const unsigned long long old = atomicAdd(&c->call_tix, 1ull);
    if ((unsigned)(old & ((1ull << kCallShift) - 1)) == gridDim.x - 1)
        atomicAdd(&c->call_tix, (1ull << kCallShift) - gridDim.x);
    return old >> kCallShift;
}

constexpr unsigned kFlagBadIndex = 1u;
constexpr unsigned kFlagTimeout = 2u;
constexpr unsigned kFlagRankStale = 4u;

// ---- rank mode: slots whose priority changed since the order was last made ------------------
// Update and insertion mark every slot they write with the current mark epoch and, the first
// time in that epoch, append it to a list of at most kMaxDirty slots together with the order key
// it had before that first write (the key it holds in the order); the next sample merges them
// into the previous order instead of sorting every slot again (k_rank.cu), then opens a new epoch,
// which unmarks every slot at once.  Null mark: nothing is marked.
constexpr unsigned kMaxDirty = 4096;

struct DirtyRefs {
    unsigned *mark;          // [capacity] the epoch in which each slot was last marked
    const unsigned *epoch;   // the current epoch (never 0, so a cleared mark is not current)
    unsigned *list;          // [kMaxDirty] marked slots
    unsigned *oldkey;        // [kMaxDirty] their order key before the first write (~bits of the raw)
    unsigned *count;         // slots marked in this epoch (the list holds the first kMaxDirty)
};

// The order key of a raw priority: raw > 0, so ascending ~bits is descending raw (an empty
// slot's 0 gives the largest key).
__device__ __forceinline__ unsigned order_key(float raw) { return ~__float_as_uint(raw); }

// Called by the one writer of `slot` in a launch, with the raw priority the slot held before
// this write.
__device__ __forceinline__ void mark_dirty(const DirtyRefs &d, unsigned long long slot, float old_raw)
{
    if (!d.mark) return;
    const unsigned e = __ldcg(d.epoch);
    if (atomicExch(&d.mark[slot], e) != e) {
        const unsigned i = atomicAdd(d.count, 1u);
        if (i < kMaxDirty) {
            d.list[i] = (unsigned)slot;
            d.oldkey[i] = order_key(old_raw);
        }
    }
}

// ---- Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11) -----------------------------------
// Round: (c0,c1,c2,c3) -> (hi(B*c2)^c1^k0, lo(B*c2), hi(A*c0)^c3^k1, lo(A*c0)) with
// A = 0xD2511F53, B = 0xCD9E8D57; the key advances by (0x9E3779B9, 0xBB67AE85) per round.
// (A loop rather than ten unrolled rounds: the kernels run it once or twice per thread, where
// code fetched once per launch costs more than the loop's count and branch.)
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint2 k)
{
#pragma unroll 1
    for (int r = 0; r < 10; ++r) {
        const unsigned a_lo = 0xD2511F53u * c.x, a_hi = __umulhi(0xD2511F53u, c.x);
        const unsigned b_lo = 0xCD9E8D57u * c.z, b_hi = __umulhi(0xCD9E8D57u, c.z);
        c = make_uint4(b_hi ^ c.y ^ k.x, b_lo, a_hi ^ c.w ^ k.y, a_lo);
        k.x += 0x9E3779B9u;
        k.y += 0xBB67AE85u;
    }
    return c;
}

// v * 2^scale for an integer 0 <= v < 2^53, assembled from bits on the integer pipe (the
// value is exact, as the binary64 conversion and scaling would give, without using GB300's
// narrow binary64 pipe).
__device__ __forceinline__ double exact_double(unsigned long long v, int scale)
{
    if (v == 0) return 0.0;
    const int p = 63 - __clzll((long long)v);
    const unsigned long long mant = (v << (52 - p)) & 0xFFFFFFFFFFFFFull;
    const unsigned long long ex = (unsigned long long)(p + scale + 1023);
    return __longlong_as_double((long long)((ex << 52) | mant));
}

// 53-bit uniform in [0, 1) of draw j in sample call `call`, stream tag `tag`.
__device__ __forceinline__ double draw_uniform(unsigned long long seed, unsigned j,
                                               unsigned long long call, unsigned tag)
{
    const uint4 x = philox4x32_10(make_uint4(j, (unsigned)call, (unsigned)(call >> 32), tag),
                                  make_uint2((unsigned)seed, (unsigned)(seed >> 32)));
    const unsigned long long bits = ((unsigned long long)x.x << 21) | (x.y >> 11);
    return exact_double(bits, -53);
}

// ---- priority transforms ("GPU-Resident Prioritized Experience Replay": Priority update,
// Error Handling & Fallback) -------------------------------------------------------------------
__device__ __forceinline__ float td_to_raw(float td, double eps, float max_at_start)
{
    if (isnan(td)) return (float)eps;
    const float a = fabsf(td);
    if (isinf(a)) return max_at_start;
    return __double2float_rn(__dadd_rn((double)a, eps));
}

__device__ __forceinline__ float prio_to_raw(float p, double eps, float max_at_start)
{
    if (isnan(p)) return (float)eps;
    if (isinf(p) && p > 0.0f) return max_at_start;
    if ((double)p < eps) return (float)eps;
    return p;
}

__device__ __forceinline__ float raw_to_leaf(float raw, double alpha)
{
    return __double2float_rn(pow((double)raw, alpha));
}

__device__ __forceinline__ float leaf_min_value(float leaf)
{
    return leaf > 0.0f ? leaf : __int_as_float(0x7f800000);
}

// ---- launch arguments --------------------------------------------------------------------
struct TreeRefs {
    float *L;
    double *S;
    float *M;
    unsigned long long n;
    int D;
};

struct RingRefs {
    float *states, *next;
    unsigned *actions;
    float *rewards;
    unsigned char *dones;
    unsigned long long capacity;
    unsigned d;
};

// Host launchers (each returns the launch's cudaError_t).
cudaError_t launch_fill_mins(float *M, unsigned long long n, cudaStream_t st);

// *marked (may be null) tells whether the insertion marked its slots (the incremental path) or
// rewrote them in bulk without marks.
cudaError_t launch_add(const TreeRefs &t, const RingRefs &r, float *raw_store, Ctl *ctl,
                       unsigned long long count, const float *states, const float *next,
                       const unsigned *actions, const float *rewards, const unsigned char *dones,
                       const float *prio, double alpha, double eps, bool proportional,
                       unsigned long long host_cursor, int num_sms, const DirtyRefs &dirty,
                       const double *rank_cdf, bool *marked, cudaStream_t st);

// A few entries (proportional mode, with a tree): one warp propagates them one after another,
// each from its leaf to the root.  Same result as launch_update.
cudaError_t launch_update_element(const TreeRefs &t, Ctl *ctl, unsigned B, const long long *idx,
                                  const float *td, double alpha, double eps, cudaStream_t st);

// Large batches: last-writer-wins scatter through the winner words `win` (one per slot, zero
// between calls), then (proportional) a rebuild of every tree level.  Same result as
// launch_update.
cudaError_t launch_update_rebuild(const TreeRefs &t, float *raw_store, Ctl *ctl, unsigned B,
                                  const long long *idx, const float *td, double alpha, double eps,
                                  bool proportional, int num_sms, const DirtyRefs &dirty, unsigned *win,
                                  const CrowdRefs &crowd, cudaStream_t st);

// P: log2 of the subtree count (-1: update_subtree_log(B, D)); at most 10 and D - 1.
cudaError_t launch_update(const TreeRefs &t, float *raw_store, Ctl *ctl, unsigned B,
                          const long long *idx, const float *td, double alpha, double eps,
                          bool proportional, int num_sms, const DirtyRefs &dirty, const CrowdRefs &crowd,
                          int P, cudaStream_t st);

constexpr int kMaxUpdateLog = 10;   // the update kernel's subtree count is at most 2^10

// log2 of the update kernel's subtree count for a batch of B entries on a tree of depth D
int update_subtree_log(unsigned B, int D);

struct SampleOut {
    long long *idx;
    float *w;
    float *states, *next;
    unsigned *actions;
    float *rewards;
    unsigned char *dones;      // uint8, or float when dones_f32
    int dones_f32;
    unsigned dp;
};

cudaError_t launch_sample_prop(const TreeRefs &t, const RingRefs &r, Ctl *ctl, unsigned B,
                               float beta, unsigned long long seed, const SampleOut &o,
                               int num_sms, cudaStream_t st);

// Uniform mode: draw j takes slot floor((j + u_j) * size / B) (counter tag 2), weight 1.
cudaError_t launch_sample_uniform(const RingRefs &r, Ctl *ctl, unsigned B, unsigned long long seed,
                                  const SampleOut &o, int num_sms, cudaStream_t st);

// Flat mode ("GPU-Resident Prioritized Experience Replay", Sampling Kernels, Proportional steps
// 2-3): the cumulative array of the leaves, rebuilt at each sample (fixed-point sums with the unit
// 2^-52 of the largest leaf's binade, rounded once to binary64), and searched by the sampler.
struct FlatWork {
    double *C;                   // [capacity] C[i] = sum of leaves 0..i (filled slots)
    unsigned long long *agg;     // [tiles] each tile's fixed-point sum
    unsigned long long *excl;    // [2 tiles] the sum of the tiles before it (128 bits: low, high)
    float *tmin;                 // [tiles] each tile's smallest filled leaf
    unsigned *tick;              // [2]: arrivals of the reduce pass
    unsigned long long *res;     // [4]: [1] T = C[size-1] (binary64 bits), [2] smallest filled leaf (bits)
};

unsigned long long flat_tiles(unsigned long long capacity);

// Rebuilds C over the filled slots; T and the smallest leaf land in res[1], res[2].
cudaError_t launch_flat_scan(const float *L, const FlatWork &fw, Ctl *ctl, unsigned long long capacity,
                             cudaStream_t st);

// Draw j (counter tag 0, as proportional mode): mass_j = (j + u_j) (T / B), the first slot with
// C[slot] > mass_j, w = (L[slot] / p_min)^-beta, fused gather.
cudaError_t launch_sample_flat(const float *L, const FlatWork &fw, const RingRefs &r, Ctl *ctl, unsigned B,
                               float beta, unsigned long long seed, const SampleOut &o, int num_sms,
                               cudaStream_t st);

// One bucket of the guide to the CDF: a mass m with fl(k delta) <= m < fl((k+1) delta) has its
// rank (the first r with cdf[r] > m) in [r0, r1], r0 the first r with cdf[r] > fl(k delta) and r1
// the first with cdf[r] > fl((k+1) delta) (capacity + 1 when none); c[i] = cdf[r0 + i] for
// i < min(r1 - r0, 3), so a bucket with at most three candidates decides the rank from its own 32
// bytes.
struct GuideEntry {
    unsigned r0, r1;
    double c[3];
};
static_assert(sizeof(GuideEntry) == 32, "one sector per guide bucket");

struct RankWork {
    float *raw;
    double *cdf;
    // guide to the CDF: guide[k] for k = 0 .. guide_k (see GuideEntry)
    GuideEntry *guide;
    unsigned guide_k;
    double guide_delta;
    unsigned *keys[2];
    unsigned *vals[2];
    unsigned *digit_hist;          // [4][256] digit counts of the sort in progress (zero between sorts)
    unsigned long long *status;    // [4][ntiles][256] look-back words: epoch | flag | count
    unsigned *sort_ctl;            // [8]: tile counters of the four passes, [4] the sort epoch
    unsigned *err;                 // device error word (PER_DEVFLAG_TIMEOUT)
    unsigned long long capacity;
    int num_sms;                   // grid of the histogram kernel
    // kept between calls by a buffer (all null for the allocation-free entry point):
    DirtyRefs dirty;               // slots changed since the order was made
    unsigned *merge_ctl;           // [8]: [1] mark epoch, [2] arrivals of the merge, [3] marked count,
                                   // [4] which of keys/vals[0|1] holds the current order
};

// Words of RankWork scratch the sort needs for `capacity` keys (beyond keys and values).
unsigned long long rank_status_words(unsigned long long capacity);

cudaError_t launch_build_cdf(double *cdf, unsigned long long capacity, double alpha,
                             cudaStream_t st);

// guide[0 .. K + 1] for a CDF of `capacity` ranks (K = guide_k, delta = guide_delta).
cudaError_t launch_build_guide(const double *cdf, unsigned long long capacity, GuideEntry *guide, unsigned K,
                               double delta, cudaStream_t st);

// Sorts the `size` filled slots by raw priority descending, ties by slot ascending, leaving
// the slot order in *sorted (a pointer into w.vals).  With keys_out non-null the last pass also
// writes the sorted keys there (*keys_out = a pointer into w.keys).
cudaError_t launch_rank_sort(RankWork &w, unsigned long long host_size, unsigned **sorted,
                             cudaStream_t st, unsigned **keys_out = nullptr);

// Brings the order up to date after at most kMaxDirty marked slots: the previous order
// (n_old entries, in the buffer pair merge_ctl[4] names) without the marked slots, merged with
// the marked slots at their current priority, into the other pair; flips merge_ctl[4] and
// clears the marks.  The full sort sets merge_ctl[4] = 1.
cudaError_t launch_rank_merge(RankWork &w, unsigned long long n_old, cudaStream_t st);

// The slot order is w.vals[merge_ctl[4]] (read on the device), or `sorted` when w.merge_ctl is null.
cudaError_t launch_sample_rank(const RankWork &w, const unsigned *sorted, const RingRefs &r,
                               Ctl *ctl, unsigned B, float beta, double alpha,
                               unsigned long long seed, const SampleOut &o, int num_sms,
                               cudaStream_t st);

unsigned long long rank_tile_count(unsigned long long capacity);

// ---- programmatic dependent launch -----------------------------------------------------------
// Every hot kernel is launched with programmatic stream serialization: its CTAs may be scheduled
// while the previous kernel in the stream is still finishing, and they wait in pdl_wait() --
// before reading any state a predecessor may write -- until that kernel has completed and its
// memory is visible.  pdl_release() lets the next kernel begin launching early.  In a kernel
// launched without the attribute both are no-ops.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_release() { asm volatile("griddepcontrol.launch_dependents;" :::); }

bool pdl_enabled();

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), unsigned grid, unsigned block, size_t smem,
                       cudaStream_t st, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl_enabled() ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// The same, with the whole grid as one thread-block cluster (grid <= 16 CTAs; the kernel must
// allow a non-portable cluster size above 8).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_cluster(void (*kernel)(KArgs...), unsigned grid, unsigned block, size_t smem,
                               cudaStream_t st, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl_enabled() ? 1 : 0;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = grid;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Every thread of every CTA of the cluster arrives (its earlier memory operations released at
// cluster scope) and waits for all the others (acquire).  A hardware barrier: no polling.
__device__ __forceinline__ void cluster_sync_all()
{
    asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

// The two halves of a cluster barrier, for a barrier whose wait can come long after the arrival:
// arrive (no memory ordering) ... wait (acquire).
__device__ __forceinline__ void cluster_arrive_relaxed()
{
    asm volatile("barrier.cluster.arrive.relaxed;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait_acquire()
{
    asm volatile("barrier.cluster.wait.acquire;" ::: "memory");
}

// The shared::cluster address of shared variable *p in the cluster's CTA `rank`.
__device__ __forceinline__ unsigned cluster_smem_addr(const void *p, unsigned rank)
{
    const unsigned s = (unsigned)__cvta_generic_to_shared(p);
    unsigned r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(s), "r"(rank));
    return r;
}

__device__ __forceinline__ void st_cluster_f64(unsigned addr, double v)
{
    asm volatile("st.shared::cluster.f64 [%0], %1;" ::"r"(addr), "d"(v) : "memory");
}

__device__ __forceinline__ void st_cluster_f32(unsigned addr, float v)
{
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

__device__ __forceinline__ void st_cluster_u32(unsigned addr, unsigned v)
{
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ unsigned cluster_cta_rank()
{
    unsigned r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Kernel attributes set once per device before the first launch (dynamic shared-memory limits
// and one common L1/shared carveout, so consecutive kernels never make an SM reconfigure).
cudaError_t init_tree_kernels(int carveout);
cudaError_t init_sample_kernels(int carveout);
cudaError_t init_rank_kernels(int carveout);

}  // namespace gbper
