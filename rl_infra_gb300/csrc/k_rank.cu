// k_rank.cu -- rank-based prioritization: the stable descending sort of (raw priority, slot)
// and the rank CDF ("GPU-Resident Prioritized Experience Replay", Sampling Kernels,
// Rank-based: sort (priority, index) pairs descending, then probabilities 1/rank^alpha and
// their cumulative sum).
//
// Sort: least-significant-digit radix sort, four passes of 8 bits over the key ~bits(raw)
// (raw > 0, so ascending ~bits is descending raw), values = slot.  One kernel counts all four
// digit histograms; each pass is then one kernel with decoupled look-back (tiles learn the
// count of earlier keys per digit from their predecessors' published words; the only waits are
// on tiles that started earlier, and each poll loop is bounded).  Pass 0 reads the raw
// priorities directly and makes the slot values on the fly; the last pass writes only the slot
// values.  Ties keep ascending slot order because every pass is stable and pass 0 starts in
// slot order.
#include "per_internal.cuh"

#include <algorithm>
#include <mutex>

namespace gbper {

namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kItems = 7;                        // keys per thread per tile
constexpr int kTile = kThreads * kItems;          // 7168: 2^20 keys are 147 tiles, one per SM
constexpr int kGroup = 16;                        // tiles per look-back group
constexpr int kMaxGroups = 16;                    // group totals read per round
constexpr unsigned kFull = 0xffffffffu;

// All four digit histograms at once: they depend on the key set, not on its order.  Every lane
// counts into its own copy of the 4 x 256 bins, laid out with a stride of 257 words, so lanes
// that meet the same digit (the high digits of floats of similar magnitude) hit distinct banks.
// Block 0 also opens a new sort epoch, which tags this sort's look-back words.
constexpr int kHistThreads = 1024;
constexpr int kHistStride = 257;
constexpr int kHistCopy = 32 * kHistStride;
constexpr size_t kHistSmem = 4ull * kHistCopy * sizeof(unsigned);   // 131,584 bytes

__global__ void __launch_bounds__(kHistThreads) k_rs_hist4(const float *raw, unsigned long long size,
                                                            unsigned *digit_hist, unsigned *sort_ctl,
                                                            unsigned *mctl)
{
    extern __shared__ unsigned s_h[];   // [4 digits][32 lanes][257]
    for (int i = threadIdx.x; i < 4 * kHistCopy; i += blockDim.x) s_h[i] = 0;
    pdl_wait();
    pdl_release();
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        atomicAdd(&sort_ctl[4], 1u);
        if (mctl) {
            // a buffer's order: the four passes leave it in keys[1] / vals[1] (mctl[4]); every
            // mark is void once every slot is sorted, so a new mark epoch opens (mctl[1]) with an
            // empty list (mctl[3])
            mctl[4] = 1u;
            mctl[1] += 1u;
            mctl[3] = 0u;
        }
    }
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const unsigned long long stride = (unsigned long long)gridDim.x * blockDim.x;
    unsigned *mine = s_h + lane * kHistStride;
    constexpr int kU = 8;   // loads in flight per thread
    for (unsigned long long p0 = (unsigned long long)blockIdx.x * blockDim.x + threadIdx.x; p0 < size;
         p0 += kU * stride) {
        unsigned k[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const unsigned long long p = p0 + u * stride;
            k[u] = p < size ? order_key(__ldg(raw + p)) : 0u;
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            if (p0 + u * stride >= size) break;
#pragma unroll
            for (int b = 0; b < 4; ++b) atomicAdd(&mine[b * kHistCopy + ((k[u] >> (8 * b)) & 255u)], 1u);
        }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < 4 * 256; i += blockDim.x) {
        const unsigned *c = s_h + (i >> 8) * kHistCopy + (i & 255);
        unsigned sum = 0;
#pragma unroll 8
        for (int l = 0; l < 32; ++l) sum += c[l * kHistStride];
        if (sum) atomicAdd(&digit_hist[i], sum);
    }
}

constexpr unsigned long long kFlagAgg = 1ull;
constexpr int kSpinLimit = 1 << 20;  // look-back poll rounds before the wait is declared lost

__device__ __forceinline__ unsigned long long status_word(unsigned epoch, unsigned long long flag,
                                                          unsigned count)
{
    return ((unsigned long long)(epoch & 0x3FFFFFFFu) << 34) | (flag << 32) | count;
}

__device__ __forceinline__ bool word_ready(unsigned long long w, unsigned want)
{
    return (unsigned)(w >> 34) == want && ((w >> 32) & 3ull) != 0;
}

// Adds the counts of the published words p[q * stride], q < count <= N, to *sum.  Every round
// re-reads all words still pending at once, so the wait costs one memory round trip beyond the
// last word's arrival.  Returns false when the rounds ran out (the sum is then incomplete).
template <int N>
__device__ __forceinline__ bool sum_published(const volatile unsigned long long *p, unsigned long long stride,
                                              unsigned count, unsigned want, unsigned *sum)
{
    unsigned pending = count >= 32 ? 0xffffffffu : ((1u << count) - 1u);
    unsigned long long w[N];
    for (int it = 0; pending && it < kSpinLimit; ++it) {
#pragma unroll
        for (int q = 0; q < N; ++q)
            if ((pending >> q) & 1u) w[q] = p[(unsigned long long)q * stride];
#pragma unroll
        for (int q = 0; q < N; ++q)
            if (((pending >> q) & 1u) && word_ready(w[q], want)) {
                *sum += (unsigned)w[q];
                pending &= ~(1u << q);
            }
    }
    return pending == 0;
}

// The digit's global start (exclusive scan of this pass's histogram row, into s_base), the sort
// epoch and the tile index.  Tiles take their index in start order, so every predecessor of a
// tile is already running.  The tile that takes the last index clears the histogram row and the
// counter for the next sort: every tile read the row before taking its index.
__device__ __forceinline__ void onesweep_prologue(int pass, unsigned ntiles, unsigned *digit_hist,
                                                  unsigned *sort_ctl, unsigned *s_base, unsigned *s_warp_tot,
                                                  unsigned *s_tile, unsigned *s_epoch)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;   // digit tid: threads 0..255
    unsigned c = 0, incl = 0;
    if (tid < 256) {
        c = digit_hist[pass * 256 + tid];
        incl = c;
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned v = __shfl_up_sync(kFull, incl, o);
            if (lane >= o) incl += v;
        }
        if (lane == 31) s_warp_tot[warp] = incl;
    }
    __syncthreads();
    if (tid < 256) {
        unsigned before = 0;
        for (int w = 0; w < warp; ++w) before += s_warp_tot[w];
        s_base[tid] = before + incl - c;
    }
    if (tid == 0) {
        *s_epoch = *(volatile unsigned *)&sort_ctl[4];
        *s_tile = atomicAdd(&sort_ctl[pass], 1u);
    }
    __syncthreads();
    if (*s_tile == ntiles - 1 && tid < 256) {
        digit_hist[pass * 256 + tid] = 0;
        if (tid == 0) sort_ctl[pass] = 0;
    }
}

// One pass of the sort (8 bits at `shift`), one kernel, one tile of 7168 keys per CTA.  A tile
// ranks its keys stably (per-warp running counts; lanes with equal digits found by bit ballots),
// publishes its digit counts, and learns how many keys of each digit precede it from two levels
// of published words: the totals of the earlier groups of 16 tiles (each published by the
// group's last tile) and the counts of the earlier tiles of its own group.  The digit's global
// start comes from the pass histogram.  The tile is staged in digit order in shared memory and
// every digit's run is written contiguously.
//
// Passes 1-3 run their prologue before waiting on the previous pass: the histogram row, the
// epoch and the tile counter were last written two or more kernels earlier (the histogram
// kernel, and the previous sort), and a kernel starts only once the kernel two places before it
// in the stream has completed.  Pass 0 reads the histogram its predecessor wrote, so it waits
// first.
__global__ void __launch_bounds__(kThreads) k_rs_onesweep(const float *raw, const unsigned *keys_in,
                                                           const unsigned *vals_in, unsigned *keys_out,
                                                           unsigned *vals_out, unsigned long long size,
                                                           int pass, unsigned ntiles, unsigned *digit_hist,
                                                           unsigned long long *status, unsigned *sort_ctl,
                                                           unsigned *err)
{
    __shared__ unsigned s_base[256];
    __shared__ unsigned s_toff[256], s_part[4][256], s_delta[256];
    __shared__ unsigned s_wcnt[kWarps][256];
    extern __shared__ unsigned s_stage[];   // the tile in digit order: keys [kTile], values [kTile]
    unsigned *s_keys = s_stage, *s_vals = s_stage + kTile;
    __shared__ unsigned s_tile, s_epoch;
    __shared__ unsigned s_warp_tot[kWarps];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int shift = 8 * pass;
    const unsigned ngroups = (ntiles + kGroup - 1) / kGroup;
    for (int i = tid; i < kWarps * 256; i += kThreads) (&s_wcnt[0][0])[i] = 0;
    if (pass > 0) {
        onesweep_prologue(pass, ntiles, digit_hist, sort_ctl, s_base, s_warp_tot, &s_tile, &s_epoch);
        pdl_wait();
    } else {
        pdl_wait();
        onesweep_prologue(pass, ntiles, digit_hist, sort_ctl, s_base, s_warp_tot, &s_tile, &s_epoch);
    }
    pdl_release();
    const unsigned tile = s_tile, epoch = s_epoch;

    // local stable ranking: warp w takes keys [w * 224, +224) of the tile in 7 rounds of 32
    const unsigned long long tbase = (unsigned long long)tile * kTile;
    const int nvalid = size - tbase < (unsigned long long)kTile ? (int)(size - tbase) : kTile;
    const int wofs = warp * (kTile / kWarps);
    const int wvalid = nvalid - wofs;       // keys of this warp: rounds i with i*32+lane < wvalid
    unsigned k[kItems], v[kItems], rk[kItems];
    const unsigned lt = (1u << lane) - 1u;
    // every key and value of the thread first, in one round of loads (the ranking loop below
    // synchronises the warp, which loads may not cross)
    {
        const unsigned long long w0 = tbase + wofs + lane;
        const unsigned *kp = keys_in ? keys_in + w0 : nullptr, *vp = vals_in ? vals_in + w0 : nullptr;
        const float *rp = raw ? raw + w0 : nullptr;
#pragma unroll
        for (int i = 0; i < kItems; ++i) {
            const bool ok = i * 32 + lane < wvalid;
            k[i] = ok ? (rp ? order_key(__ldg(rp + i * 32)) : __ldg(kp + i * 32)) : 0u;
            v[i] = ok ? (rp ? (unsigned)(w0 + i * 32) : __ldg(vp + i * 32)) : 0u;
        }
    }
    // lanes with each key's digit: one ballot per digit bit and one for validity, for all rounds
    // first (independent of one another), then one shared-memory atomic per digit and round by
    // the digit's lowest lane, whose result (the warp's count of that digit so far) is broadcast
    unsigned pm[kItems];
#pragma unroll
    for (int i = 0; i < kItems; ++i) {
        const bool ok = i * 32 + lane < wvalid;
        const unsigned dg = (k[i] >> shift) & 255u;
        unsigned peers = __ballot_sync(kFull, ok);
        if (!ok) peers = ~peers;
#pragma unroll
        for (int b = 0; b < 8; ++b) {
            const unsigned ones = 0u - ((dg >> b) & 1u);    // all ones where the bit is set
            const unsigned bb = __ballot_sync(kFull, ones);
            peers &= ~(bb ^ ones);
        }
        pm[i] = peers;
    }
#pragma unroll
    for (int i = 0; i < kItems; ++i) {
        const bool ok = i * 32 + lane < wvalid;
        const unsigned dg = (k[i] >> shift) & 255u;
        const int leader = __ffs(pm[i]) - 1;
        unsigned old = 0;
        if (ok && lane == leader) old = atomicAdd(&s_wcnt[warp][dg], (unsigned)__popc(pm[i]));
        old = __shfl_sync(kFull, old, leader);
        rk[i] = old + __popc(pm[i] & lt);
        __syncwarp();
    }
    __syncthreads();
    // this tile's count of each digit, published at once (four threads per digit add eight
    // warps' counts each); then the start of each digit's run within the tile and of each
    // warp's share of it, and the tile staged in digit order in shared memory
    unsigned long long *row = status + ((unsigned long long)pass * ntiles) * 256;
    unsigned long long *grow = status + 4ull * ntiles * 256 + (unsigned long long)pass * ngroups * 256;
    volatile unsigned long long *vrow = row, *vgrow = grow;
    const unsigned want = epoch & 0x3FFFFFFFu;
    const int d = tid & 255, quarter = tid >> 8;
    {
        unsigned c = 0;
#pragma unroll
        for (int w = 0; w < kWarps / 4; ++w) c += s_wcnt[quarter * (kWarps / 4) + w][d];
        s_part[quarter][d] = c;
    }
    __syncthreads();
    unsigned cnt = 0, inc = 0;
    if (tid < 256) {
        cnt = s_part[0][d] + s_part[1][d] + s_part[2][d] + s_part[3][d];
        vrow[(unsigned long long)tile * 256 + d] = status_word(epoch, kFlagAgg, cnt);
        inc = cnt;
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned x = __shfl_up_sync(kFull, inc, o);
            if (lane >= o) inc += x;
        }
        if (lane == 31) s_warp_tot[warp] = inc;
    }
    __syncthreads();
    {
        // exclusive start of digit d within the tile (each quarter redoes the warp scan of its
        // 32 digits), then of the first of this quarter's eight warps within the digit's run
        unsigned bef = 0;
        for (int w = 0; w < (d >> 5); ++w) bef += s_warp_tot[w];
        const unsigned cd = s_part[0][d] + s_part[1][d] + s_part[2][d] + s_part[3][d];
        unsigned in = cd;
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned x = __shfl_up_sync(kFull, in, o);
            if (lane >= o) in += x;
        }
        const unsigned dx = bef + in - cd;
        unsigned run = dx;
        for (int q = 0; q < quarter; ++q) run += s_part[q][d];
#pragma unroll
        for (int w = 0; w < kWarps / 4; ++w) {
            const int ww = quarter * (kWarps / 4) + w;
            const unsigned cw = s_wcnt[ww][d];
            s_wcnt[ww][d] = run;
            run += cw;
        }
        if (tid < 256) s_toff[d] = dx;
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < kItems; ++i) {
        if (i * 32 + lane < wvalid) {
            const unsigned dg = (k[i] >> shift) & 255u;
            const unsigned tpos = s_wcnt[warp][dg] + rk[i];
            s_keys[tpos] = k[i];
            s_vals[tpos] = v[i];
        }
    }
    // keys of digit d in earlier tiles: the counts of the earlier tiles of this tile's group
    // (quarter 0) plus the totals of the earlier complete groups of kGroup tiles (quarter 1)
    const unsigned grp = tile / kGroup, first = grp * kGroup;
    bool ok = true;
    unsigned part = 0;
    if (quarter == 0) {
        if (tile % kGroup == kGroup - 1) {  // the last tile of a group publishes the group total
            unsigned gsum = cnt;
            ok &= sum_published<kGroup - 1>(vrow + (unsigned long long)first * 256 + d, 256, kGroup - 1, want, &gsum);
            vgrow[(unsigned long long)grp * 256 + d] = status_word(epoch, kFlagAgg, gsum);
            part = gsum - cnt;
        } else {
            ok &= sum_published<kGroup - 1>(vrow + (unsigned long long)first * 256 + d, 256, tile - first, want, &part);
        }
    } else if (quarter == 1) {
        for (unsigned q0 = 0; q0 < grp; q0 += kMaxGroups) {
            const unsigned m = grp - q0 < kMaxGroups ? grp - q0 : kMaxGroups;
            ok &= sum_published<kMaxGroups>(vgrow + (unsigned long long)q0 * 256 + d, 256, m, want, &part);
        }
    }
    if (!ok) atomicOr(err, kFlagTimeout);  // a wait gave up: this sort's output is not valid
    if (quarter == 1) s_part[1][d] = part;   // s_part was last read before the staging barrier
    __syncthreads();
    // output position of staged key t of digit d: s_delta[d] + t
    if (quarter == 0) s_delta[d] = s_base[d] + s_part[1][d] + part - s_toff[d];
    __syncthreads();
    for (int t = tid; t < nvalid; t += kThreads) {
        const unsigned key = s_keys[t];
        const unsigned pos = s_delta[(key >> shift) & 255u] + (unsigned)t;
        if (keys_out) keys_out[pos] = key;
        vals_out[pos] = s_vals[t];
    }
}

// c[r] = sum_{k<=r} k^-alpha for r in [0, C]: each thread sums a contiguous chunk with
// compensated (Kahan) summation, one thread adds the chunk totals in order, and every thread
// then writes its chunk's running values.
__global__ void __launch_bounds__(1024) k_build_cdf(double *cdf, unsigned long long C, double alpha)
{
    __shared__ double s_tot[1024];
    const unsigned long long per = (C + blockDim.x - 1) / blockDim.x;
    const unsigned long long k0 = 1 + threadIdx.x * per;
    const unsigned long long k1 = min(k0 + per, C + 1);
    double sum = 0.0, comp = 0.0;
    for (unsigned long long k = k0; k < k1; ++k) {
        const double term = pow((double)k, -alpha);
        const double y = __dsub_rn(term, comp);
        const double t = __dadd_rn(sum, y);
        comp = __dsub_rn(__dsub_rn(t, sum), y);
        sum = t;
    }
    s_tot[threadIdx.x] = sum;
    __syncthreads();
    if (threadIdx.x == 0) {
        double run = 0.0;
        for (unsigned i = 0; i < blockDim.x; ++i) {
            const double v = s_tot[i];
            s_tot[i] = run;
            run = __dadd_rn(run, v);
        }
        cdf[0] = 0.0;
    }
    __syncthreads();
    sum = s_tot[threadIdx.x];
    comp = 0.0;
    for (unsigned long long k = k0; k < k1; ++k) {
        const double term = pow((double)k, -alpha);
        const double y = __dsub_rn(term, comp);
        const double t = __dadd_rn(sum, y);
        comp = __dsub_rn(__dsub_rn(t, sum), y);
        sum = t;
        cdf[k] = sum;
    }
}

// The first r in [1, C] with cdf[r] > thr (C + 1 if none).
__device__ __forceinline__ unsigned long long cdf_first_above(const double *cdf, unsigned long long C, double thr)
{
    unsigned long long lo = 1, hi = C + 1;
    while (lo < hi) {
        const unsigned long long mid = lo + (hi - lo) / 2;
        if (cdf[mid] > thr) hi = mid;
        else lo = mid + 1;
    }
    return lo;
}

// guide[k], k = 0 .. K (see GuideEntry): r0 and r1 from the thresholds fl(k * delta) and
// fl((k + 1) * delta), formed with the same binary64 products as the sampler's (r1 = C + 1 for
// the last bucket).
__global__ void k_build_guide(const double *cdf, unsigned long long C, GuideEntry *guide, unsigned K, double delta)
{
    for (unsigned long long k = blockIdx.x * (unsigned long long)blockDim.x + threadIdx.x; k <= (unsigned long long)K;
         k += (unsigned long long)gridDim.x * blockDim.x) {
        GuideEntry g;
        const unsigned long long r0 = cdf_first_above(cdf, C, __dmul_rn((double)k, delta));
        const unsigned long long r1 = k == K ? C + 1 : cdf_first_above(cdf, C, __dmul_rn((double)(k + 1), delta));
        g.r0 = (unsigned)r0;
        g.r1 = (unsigned)r1;
        for (int i = 0; i < 3; ++i) g.c[i] = r0 + i < r1 && r0 + i <= C ? cdf[r0 + i] : 0.0;
        guide[k] = g;
    }
}

// ------------------------------------------------------------------------------------------
// Incremental order: between two samples only the slots that update and insertion wrote have a
// new priority; each is listed once, with the key it held in the order.  The new order is the
// previous order without those slots' old entries, merged with their new entries -- the same
// sequence a full sort gives, since the order is a total order on (key, slot).  One kernel, one
// 8192-entry tile of the previous order per CTA, no CTA waiting for another.  Every listed slot
// gives an old entry (old key, slot), which is an entry of the previous order, and a new entry
// (current key, slot).  With `lo` the previous tile's last entry and `x_last` this tile's:
//   1. the CTA stages its tile in shared memory (asynchronous 16-byte copies); it reads the listed slots: c_old = old entries at or below lo, c_new = new
//      entries at or below lo, the dropped entries (old entries in (lo, x_last]: they are in this
//      tile) and the own new entries (in (lo, x_last], or above lo for the last tile);
//   2. each dropped entry is located in the tile by binary search and marked in a bitmap of the
//      tile's 8192 entries (with per-word prefix counts, the dropped entries below any index are
//      one lookup away: they need no sort, which matters because the top ranks, where the draws
//      concentrate, collect most of them); the own new entries (few, spread like the order) are
//      located as they are found (i tile entries lie below an own entry) and sorted with that
//      count;
//   3. the tile's output starts at base = t0 - c_old + c_new (t0 entries of the previous order
//      lie at or below lo, c_old of them dropped, and c_new new entries precede the tile).  Tile
//      entry e, unless dropped, goes to e - (dropped below e) + (own with i <= e); own entry j
//      goes to i_j - (dropped below i_j) + j.  The stores are coalesced between those few
//      break points;
//   4. the last CTA to finish opens a new mark epoch (which unmarks every slot) and flips the
//      buffer pair.
// ------------------------------------------------------------------------------------------
constexpr int kMThreads = 512;                               // 16 warps: registers enough for no spills
constexpr int kMItems = 16;
constexpr int kMTile = kMThreads * kMItems;                  // 8192
constexpr int kMPre = 2;   // listed slots per thread loaded with the tile (more are read after)
constexpr int kMWords = kMTile / 32;                         // words of the tile's dropped bitmap
static_assert(kMTile % 4 == 0, "the tile's slot array must start 16 bytes after a multiple");
constexpr size_t kMergeSmem = (size_t)kMTile * 2 * sizeof(unsigned)             // the tile: keys, slots
                              + (size_t)kMaxDirty * sizeof(unsigned long long)  // own new entries
                              + (size_t)kMaxDirty * sizeof(unsigned)            // their places in the tile
                              + (size_t)2 * (kMWords + 1) * sizeof(unsigned)    // dropped bitmap, prefix counts
                              + (size_t)(kMWords + 2) * sizeof(unsigned)        // own entries before each word
                              + (size_t)(kMWords + 1) * sizeof(uint4);          // the three per word, packed

__device__ __forceinline__ unsigned long long pack_key_slot(unsigned key, unsigned slot)
{
    return ((unsigned long long)key << 32) | slot;
}

// entries of a[0, n) (ascending) that are < x
template <typename T>
__device__ __forceinline__ unsigned count_below(const T *a, unsigned n, T x)
{
    unsigned lo = 0, hi = n;
    while (lo < hi) {
        const unsigned mid = (lo + hi) >> 1;
        if (a[mid] < x) lo = mid + 1;
        else hi = mid;
    }
    return lo;
}

// entries of the staged tile (keys tk[], slots tv[], ascending as pairs) that are < x
__device__ __forceinline__ unsigned tile_below(const unsigned *tk, const unsigned *tv, unsigned n,
                                               unsigned long long x)
{
    unsigned lo = 0, hi = n;
    while (lo < hi) {
        const unsigned mid = (lo + hi) >> 1;
        if (pack_key_slot(tk[mid], tv[mid]) < x) lo = mid + 1;
        else hi = mid;
    }
    return lo;
}

// 16 bytes global -> shared without passing through registers (L2 only)
__device__ __forceinline__ void cp_async16(void *smem, const void *gmem)
{
    const unsigned sa = (unsigned)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sa), "l"(gmem) : "memory");
}

// Sorts a[0, n) ascending, carrying p[0, n) along, n <= kMaxDirty: one warp's shuffles up to 32
// entries (warp `w` of the CTA), else the CTA (every thread must call it with the same n).
__device__ __forceinline__ void sort_small(unsigned long long *a, unsigned *p, unsigned n, int w)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (n <= 32) {
        if (warp == w) {
            unsigned long long x = (unsigned)lane < n ? a[lane] : ~0ull;
            unsigned px = (unsigned)lane < n ? p[lane] : 0u;
            const unsigned lim = n <= 8 ? 8u : (n <= 16 ? 16u : 32u);   // lanes past n hold the largest key
            for (unsigned kk = 2; kk <= lim; kk <<= 1)
                for (unsigned j = kk >> 1; j > 0; j >>= 1) {
                    const unsigned long long y = __shfl_xor_sync(kFull, x, j);
                    const unsigned py = __shfl_xor_sync(kFull, px, j);
                    const bool lower = (lane & j) == 0, up = (lane & kk) == 0;
                    if (lower == up ? y < x : y > x) {
                        x = y;
                        px = py;
                    }
                }
            if ((unsigned)lane < n) {
                a[lane] = x;
                p[lane] = px;
            }
        }
        return;
    }
    unsigned m2 = 64;
    while (m2 < n) m2 <<= 1;
    for (unsigned i = n + tid; i < m2; i += blockDim.x) a[i] = ~0ull;
    __syncthreads();
    for (unsigned kk = 2; kk <= m2; kk <<= 1)
        for (unsigned j = kk >> 1; j > 0; j >>= 1) {
            for (unsigned i = tid; i < m2; i += blockDim.x) {
                const unsigned l = i ^ j;
                if (l > i) {
                    const unsigned long long x = a[i], y = a[l];
                    if ((i & kk) == 0 ? x > y : x < y) {
                        a[i] = y;
                        a[l] = x;
                        const unsigned t = p[i];
                        p[i] = p[l];
                        p[l] = t;
                    }
                }
            }
            __syncthreads();
        }
}

__global__ void __launch_bounds__(kMThreads) k_rank_merge(const float *raw, unsigned *keys0, unsigned *keys1,
                                                           unsigned *vals0, unsigned *vals1, unsigned long long n_old,
                                                           DirtyRefs dirty, unsigned *mctl, unsigned *err)
{
    extern __shared__ __align__(16) unsigned long long s_m[];
    // the tile first: the asynchronous copies write it 16 bytes at a time, at 16-byte offsets
    unsigned *tk = reinterpret_cast<unsigned *>(s_m), *tv = tk + kMTile;   // [kMTile] each: the tile
    unsigned long long *nl = reinterpret_cast<unsigned long long *>(tv + kMTile);   // [kMaxDirty] own new entries
    unsigned *nins = reinterpret_cast<unsigned *>(nl + kMaxDirty);   // [kMaxDirty] tile entries below each
    unsigned *dbits = nins + kMaxDirty;                   // [kMWords + 1] dropped tile entries
    unsigned *dpre = dbits + kMWords + 1;                 // [kMWords + 1] dropped entries in earlier words
    unsigned *ipre = dpre + kMWords + 1;                  // [kMWords + 2] own entries placed in each word, then before it
    uint4 *winfo = reinterpret_cast<uint4 *>(ipre + kMWords + 2);   // [kMWords + 1] dbits, dpre, ipre, next ipre
    __shared__ unsigned s_nn;
    __shared__ unsigned s_wo[kMThreads / 32], s_wn[kMThreads / 32], s_wd[kMWords / 32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) s_nn = 0;
    for (int i = tid; i <= kMWords; i += kMThreads) dbits[i] = 0u;
    for (int i = tid; i <= kMWords + 1; i += kMThreads) ipre[i] = 0u;
    pdl_wait();
    pdl_release();
    const unsigned tile = blockIdx.x;
    // thread 0 reads the control words for the CTA and then arrives on a ticket (the values are
    // in hand before the arrival is issued); the last CTA to have read them opens a new mark epoch
    // (which unmarks every slot), empties the list and flips the buffer pair at its end, which the
    // kernels after this one see once every CTA's output is complete
    __shared__ unsigned s_ctl[2];
    if (tid == 0) {
        s_ctl[0] = *(volatile unsigned *)dirty.count;
        s_ctl[1] = *(volatile unsigned *)&mctl[4] & 1u;
    }
    __syncthreads();
    const unsigned cnt = s_ctl[0], cur = s_ctl[1];
    const unsigned arrival = tid == 0 ? atomicAdd(&mctl[2], 1u) : 0u;   // awaited only at the end
    const unsigned *keys_in = cur ? keys1 : keys0, *vals_in = cur ? vals1 : vals0;
    unsigned *keys_out = cur ? keys0 : keys1, *vals_out = cur ? vals0 : vals1;
    const bool over = cnt > kMaxDirty;   // more slots than listed: the order cannot be merged
    if (!over) {
        const unsigned long long t0 = (unsigned long long)tile * kMTile;
        const int nt = (int)(n_old - t0 < (unsigned long long)kMTile ? n_old - t0 : (unsigned long long)kMTile);
        const bool first = tile == 0, lastt = tile + 1 == gridDim.x;
        // 1. the tile into shared memory (asynchronous 16-byte copies), its boundary entries and
        //    this thread's listed slots
#pragma unroll
        for (int c = 0; c < kMItems / 4; ++c) {
            const int e = (c * kMThreads + tid) * 4;
            if (e + 4 <= nt) {
                cp_async16(tk + e, keys_in + t0 + e);
                cp_async16(tv + e, vals_in + t0 + e);
            } else {
                for (int i = e; i < nt; ++i) {
                    tk[i] = __ldg(keys_in + t0 + i);
                    tv[i] = __ldg(vals_in + t0 + i);
                }
            }
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
        const unsigned long long lo = first ? 0ull : pack_key_slot(__ldg(keys_in + t0 - 1), __ldg(vals_in + t0 - 1));
        const unsigned long long x_last = pack_key_slot(__ldg(keys_in + t0 + nt - 1), __ldg(vals_in + t0 + nt - 1));
        unsigned ls[kMPre], lk[kMPre], lr[kMPre];
#pragma unroll
        for (int q = 0; q < kMPre; ++q) {
            const unsigned i = tid + q * kMThreads;
            ls[q] = i < cnt ? dirty.list[i] : 0u;
            lk[q] = i < cnt ? dirty.oldkey[i] : 0u;
        }
#pragma unroll
        for (int q = 0; q < kMPre; ++q) lr[q] = tid + q * kMThreads < cnt ? order_key(raw[ls[q]]) : 0u;
        asm volatile("cp.async.wait_group 0;" ::: "memory");
        __syncthreads();   // the staged tile, s_nn, the cleared bitmap
        // 2. the listed slots: counts at or below lo, dropped entries marked at their index,
        //    own new entries collected
        unsigned c_old = 0, c_new = 0;
        for (unsigned i = tid; i < cnt; i += kMThreads) {
            const int q = (int)(i / kMThreads);
            unsigned slot, okey, nkey;
            if (q < kMPre) {
                slot = q == 0 ? ls[0] : ls[1];
                okey = q == 0 ? lk[0] : lk[1];
                nkey = q == 0 ? lr[0] : lr[1];
            } else {
                slot = dirty.list[i];
                okey = dirty.oldkey[i];
                nkey = order_key(raw[slot]);
            }
            const unsigned long long xo = pack_key_slot(okey, slot);
            const unsigned long long xn = pack_key_slot(nkey, slot);
            if (!first && xo <= lo) {
                ++c_old;
            } else if (xo <= x_last) {   // an entry of this tile
                const unsigned d = tile_below(tk, tv, (unsigned)nt, xo);
                atomicOr(&dbits[d >> 5], 1u << (d & 31));
            }
            if (!first && xn <= lo) {
                ++c_new;
            } else if (lastt || xn <= x_last) {   // own: with the count of tile entries below it
                const unsigned j = atomicAdd(&s_nn, 1u);
                nl[j] = xn;
                const unsigned ij = tile_below(tk, tv, (unsigned)nt, xn);
                nins[j] = ij;
                atomicAdd(&ipre[ij >> 5], 1u);
            }
        }
        for (int o = 16; o > 0; o >>= 1) {
            c_old += __shfl_xor_sync(kFull, c_old, o);
            c_new += __shfl_xor_sync(kFull, c_new, o);
        }
        if (lane == 0) {
            s_wo[warp] = c_old;
            s_wn[warp] = c_new;
        }
        __syncthreads();   // dropped bitmap, own list, partial counts
        const unsigned nn = s_nn;
        if (warp < kMWords / 32) {   // prefix counts of the dropped bitmap, 32 words per warp
            const unsigned c = __popc(dbits[warp * 32 + lane]);
            unsigned inc = c;
            for (int o = 1; o < 32; o <<= 1) {
                const unsigned x = __shfl_up_sync(kFull, inc, o);
                if (lane >= o) inc += x;
            }
            dpre[warp * 32 + lane] = inc - c;   // within the warp's 32 words, fixed up below
            if (lane == 31) s_wd[warp] = inc;
        }
        // the CTA's counts: lane l takes warp l's partial counts, then a warp sum
        c_old = lane < kMThreads / 32 ? s_wo[lane] : 0u;
        c_new = lane < kMThreads / 32 ? s_wn[lane] : 0u;
        for (int o = 16; o > 0; o >>= 1) {
            c_old += __shfl_xor_sync(kFull, c_old, o);
            c_new += __shfl_xor_sync(kFull, c_new, o);
        }
        __syncthreads();   // the warps' bitmap totals
        if (warp < kMWords / 32) {
            unsigned before = 0;
            for (int w = 0; w < warp; ++w) before += s_wd[w];
            dpre[warp * 32 + lane] += before;
            if (warp == kMWords / 32 - 1 && lane == 31) dpre[kMWords] = before + s_wd[warp];
        }
        sort_small(nl, nins, nn, kMWords / 32);   // a warp that does not build the prefix, when short
        if (warp == kMWords / 32 + 1) {   // another: own entries placed before each word (9 words a lane)
            constexpr int kPer = (kMWords + 1 + 31) / 32;
            unsigned v[kPer], s = 0;
#pragma unroll
            for (int k = 0; k < kPer; ++k) {
                const int wi = lane * kPer + k;
                v[k] = wi <= kMWords ? ipre[wi] : 0u;
                s += v[k];
            }
            unsigned inc = s;
            for (int o = 1; o < 32; o <<= 1) {
                const unsigned x = __shfl_up_sync(kFull, inc, o);
                if (lane >= o) inc += x;
            }
            unsigned run = inc - s;
#pragma unroll
            for (int k = 0; k < kPer; ++k) {
                const int wi = lane * kPer + k;
                if (wi <= kMWords) ipre[wi] = run;
                run += v[k];
            }
            if (lane == 31) ipre[kMWords + 1] = inc;
        }
        __syncthreads();   // dpre, ipre, own entries sorted with their places
        for (int wi = tid; wi <= kMWords; wi += kMThreads)   // one 16-byte read a word in the copy below
            winfo[wi] = make_uint4(dbits[wi], dpre[wi], ipre[wi], ipre[wi + 1]);
        __syncthreads();
        // 3. the tile's output from base = t0 - c_old + c_new
        const unsigned long long base = t0 - c_old + c_new;
        // own entries at or below tile entry e: those placed in earlier words, and those of e's word
        // (a contiguous stretch of the sorted places, rarely more than one) compared one by one
#pragma unroll
        for (int q = 0; q < kMItems; ++q) {
            const unsigned e = tid + q * kMThreads;
            if ((int)e >= nt) break;
            const uint4 wf = winfo[e >> 5];   // the same word for the whole warp
            const unsigned wd = wf.x, bit = 1u << (e & 31);
            if (wd & bit) continue;   // dropped
            unsigned sn = wf.z;
            for (unsigned j = wf.z; j < wf.w; ++j) sn += nins[j] <= e ? 1u : 0u;
            const unsigned sd = wf.y + __popc(wd & (bit - 1u));
            const unsigned long long o = base + e - sd + sn;
            keys_out[o] = tk[e];
            vals_out[o] = tv[e];
        }
        for (unsigned j = tid; j < nn; j += kMThreads) {
            const unsigned i = nins[j];
            const unsigned sd = dpre[i >> 5] + __popc(dbits[i >> 5] & ((1u << (i & 31)) - 1u));
            const unsigned long long o = base + i - sd + j;
            const unsigned long long y = nl[j];
            keys_out[o] = (unsigned)(y >> 32);
            vals_out[o] = (unsigned)y;
        }
    } else if (tid == 0 && tile == 0) {
        atomicOr(err, kFlagRankStale);
    }
    if (tid == 0 && arrival == gridDim.x - 1) {
        if (cnt <= kMaxDirty) {
            *dirty.count = 0u;
            mctl[1] += 1u;
            mctl[4] = cur ^ 1u;   // the merged order is in the other pair
        }
        mctl[2] = 0u;
    }
}

constexpr size_t kStageSmem = 2ull * kTile * sizeof(unsigned);

// Dynamic shared-memory limits of the sort kernels, set once per device (the sort is also
// reached without a buffer, through per_rank_order_noalloc).
std::mutex g_attr_mu;
bool g_attr_done[64] = {};

cudaError_t ensure_sort_attributes()
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_attr_mu);
    if (g_attr_done[dev]) return cudaSuccess;
    e = cudaFuncSetAttribute(k_rs_hist4, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kHistSmem);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(k_rank_merge, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kMergeSmem);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(k_rs_onesweep, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kStageSmem);
    if (e == cudaSuccess) g_attr_done[dev] = true;
    return e;
}

}  // namespace

cudaError_t init_rank_kernels(int carveout)
{
    cudaError_t e = ensure_sort_attributes();
    if (e != cudaSuccess || carveout < 0) return e;
    const void *fns[] = {(const void *)k_rs_hist4, (const void *)k_rs_onesweep, (const void *)k_build_cdf};
    for (const void *f : fns) {
        e = cudaFuncSetAttribute(f, cudaFuncAttributePreferredSharedMemoryCarveout, carveout);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t launch_rank_merge(RankWork &w, unsigned long long n_old, cudaStream_t st)
{
    cudaError_t e = ensure_sort_attributes();
    if (e != cudaSuccess) return e;
    const unsigned ntiles = (unsigned)std::max<unsigned long long>((n_old + kMTile - 1) / kMTile, 1);
    return launch_pdl(k_rank_merge, ntiles, kMThreads, kMergeSmem, st, (const float *)w.raw, w.keys[0], w.keys[1],
                      w.vals[0], w.vals[1], n_old, w.dirty, w.merge_ctl, w.err);
}

cudaError_t launch_build_guide(const double *cdf, unsigned long long capacity, GuideEntry *guide, unsigned K,
                               double delta, cudaStream_t st)
{
    const unsigned grid = (unsigned)std::min<unsigned long long>(((unsigned long long)K + 1 + 255) / 256, 4096);
    k_build_guide<<<grid, 256, 0, st>>>(cdf, capacity, guide, K, delta);
    return cudaGetLastError();
}

unsigned long long rank_tile_count(unsigned long long capacity)
{
    return (capacity + kTile - 1) / kTile;
}

cudaError_t launch_build_cdf(double *cdf, unsigned long long capacity, double alpha, cudaStream_t st)
{
    k_build_cdf<<<1, 1024, 0, st>>>(cdf, capacity, alpha);
    return cudaGetLastError();
}

unsigned long long rank_status_words(unsigned long long capacity)
{
    const unsigned long long t = rank_tile_count(capacity);
    return 4ull * (t + (t + kGroup - 1) / kGroup) * 256ull;
}

cudaError_t launch_rank_sort(RankWork &w, unsigned long long host_size, unsigned **sorted, cudaStream_t st,
                             unsigned **keys_out)
{
    const unsigned long long size = host_size;
    const unsigned ntiles = (unsigned)std::max<unsigned long long>(rank_tile_count(size), 1);
    cudaError_t e = ensure_sort_attributes();
    if (e != cudaSuccess) return e;
    const unsigned hgrid = (unsigned)std::min<unsigned long long>((size + kHistThreads - 1) / kHistThreads,
                                                                  (unsigned long long)std::max(w.num_sms, 1));
    e = launch_pdl(k_rs_hist4, std::max(hgrid, 1u), kHistThreads, kHistSmem, st, (const float *)w.raw, size,
                   w.digit_hist, w.sort_ctl, w.merge_ctl);
    if (e != cudaSuccess) return e;
    const unsigned *kin = nullptr, *vin = nullptr;
    int cur = 0;
    for (int pass = 0; pass < 4; ++pass) {
        const float *raw = pass == 0 ? w.raw : nullptr;
        unsigned *kout = pass == 3 && !keys_out ? nullptr : w.keys[cur];
        unsigned *vout = w.vals[cur];
        e = launch_pdl(k_rs_onesweep, ntiles, kThreads, kStageSmem, st, raw, kin, vin, kout, vout, size, pass, ntiles,
                       w.digit_hist, (unsigned long long *)w.status, w.sort_ctl, w.err);
        if (e != cudaSuccess) return e;
        kin = w.keys[cur];
        vin = w.vals[cur];
        cur ^= 1;
    }
    *sorted = const_cast<unsigned *>(vin);
    if (keys_out) *keys_out = const_cast<unsigned *>(kin);
    return cudaSuccess;
}

}  // namespace gbper

// ------------------------------------------------------------------------------------------
// per_rank_order_noalloc: the same descending sort for callers that may not allocate device
// memory.  Its scratch (key and value ping-pong buffers, digit histograms, control words and
// look-back words) is a file-scope device array of fixed size, resolved to a device address
// once per device.
// ------------------------------------------------------------------------------------------
#include "gbper.h"

#include <mutex>

namespace gbper {
namespace {

constexpr unsigned long long kNoAllocMaxKeys = 1ull << 18;
constexpr unsigned long long kNoAllocTiles = (kNoAllocMaxKeys + kTile - 1) / kTile;
constexpr unsigned long long kNoAllocGroups = (kNoAllocTiles + kGroup - 1) / kGroup;
// keys[2], values[2], digit histograms [1024], sort control [16], then 64-bit look-back words
constexpr unsigned long long kNoAllocWords =
    4 * kNoAllocMaxKeys + 1024 + 16 + 2 * (4 * (kNoAllocTiles + kNoAllocGroups) * 256);
constexpr int kNoAllocMaxDevices = 64;

// About 4.3 MiB per device, held by every device that loads the library until exit.  Zero at
// load; the look-back words rely on that (each sort tags them with a new epoch, so a word left
// by an earlier call never reads as this call's).  The histograms, tile counters and error word
// are cleared by every call.
__device__ __align__(256) unsigned g_noalloc_scratch[kNoAllocWords];

std::mutex g_noalloc_mu;
unsigned *g_noalloc_ptr[kNoAllocMaxDevices] = {};

// Device address of g_noalloc_scratch on the current device (host code cannot use the symbol
// itself: on the host it names a stand-in, not device memory).
cudaError_t noalloc_scratch(unsigned **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kNoAllocMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_noalloc_ptr[dev] = static_cast<unsigned *>(p);
    }
    *out = g_noalloc_ptr[dev];
    return cudaSuccess;
}

// Copies the sorted slots to the caller's order and reports the sort's error word: when a
// look-back wait gave up, every entry becomes 0xFFFFFFFF (no valid slot) instead of a wrong
// order, and *status (if given) receives the flag bits.  Launched without programmatic
// serialization, so it starts once the last sort pass has completed.
__global__ void k_noalloc_emit(const unsigned *sorted, unsigned n, const unsigned *err, unsigned *order,
                               unsigned *status)
{
    const unsigned flags = *(const volatile unsigned *)err;
    const unsigned i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) order[i] = flags ? 0xFFFFFFFFu : sorted[i];
    if (status && i == 0) *status = flags;
}

}  // namespace

}  // namespace gbper

extern "C" per_status per_rank_order_noalloc(const float *d_raw, uint32_t n, uint32_t *d_order,
                                             uint32_t *d_status, void *stream)
{
    using namespace gbper;
    if (!d_raw || !d_order || n == 0 || n > kNoAllocMaxKeys) return PER_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(d_raw) % 4 || reinterpret_cast<uintptr_t>(d_order) % 4 ||
        reinterpret_cast<uintptr_t>(d_status) % 4)
        return PER_ERR_INVALID_ARG;
    unsigned *base = nullptr;
    if (noalloc_scratch(&base) != cudaSuccess) {
        cudaGetLastError();
        return PER_ERR_CUDA;
    }
    RankWork w{};
    w.raw = const_cast<float *>(d_raw);
    w.keys[0] = base;
    w.keys[1] = base + kNoAllocMaxKeys;
    w.vals[0] = base + 2 * kNoAllocMaxKeys;
    w.vals[1] = base + 3 * kNoAllocMaxKeys;
    w.digit_hist = base + 4 * kNoAllocMaxKeys;
    w.sort_ctl = w.digit_hist + 1024;   // [0..3] tile counters, [4] epoch, [8] error word
    w.err = w.sort_ctl + 8;
    w.status = reinterpret_cast<unsigned long long *>(w.sort_ctl + 16);  // 8-byte aligned
    w.capacity = n;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&w.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        return PER_ERR_CUDA;
    }
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    // A call that stopped part way (a failed launch, a captured call never replayed) may have
    // left histogram counts, tile counters or the error word set: clear them (the epoch in
    // sort_ctl[4] stays, it tags this sort's look-back words).  cudaMemsetAsync allocates nothing.
    cudaError_t e = cudaMemsetAsync(w.digit_hist, 0, (1024 + 4) * sizeof(unsigned), st);
    if (e == cudaSuccess) e = cudaMemsetAsync(w.err, 0, sizeof(unsigned), st);
    unsigned *sorted = nullptr;
    if (e == cudaSuccess) e = launch_rank_sort(w, n, &sorted, st);
    if (e == cudaSuccess) {
        k_noalloc_emit<<<(n + 255) / 256, 256, 0, st>>>(sorted, n, w.err, d_order, d_status);
        e = cudaGetLastError();
    }
    if (e != cudaSuccess) cudaGetLastError();
    return e == cudaSuccess ? PER_OK : PER_ERR_CUDA;
}
