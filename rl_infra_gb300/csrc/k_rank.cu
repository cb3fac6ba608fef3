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

namespace gbper {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kItems = 16;                       // keys per thread per tile
constexpr int kTile = kThreads * kItems;          // 4096
constexpr int kGroup = 16;                        // tiles per look-back group
constexpr int kMaxGroups = 16;                    // group totals read per round
constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ unsigned key_of_raw(float raw) { return ~__float_as_uint(raw); }

// All four digit histograms at once: they depend on the key set, not on its order.  Block 0
// also opens a new sort epoch, which tags this sort's look-back words.
__global__ void __launch_bounds__(kThreads) k_rs_hist4(const float *raw, unsigned long long size,
                                                        unsigned *digit_hist, unsigned *sort_ctl)
{
    __shared__ unsigned s_h[4 * 256];
    for (int i = threadIdx.x; i < 4 * 256; i += blockDim.x) s_h[i] = 0;
    pdl_wait();
    pdl_release();
    if (blockIdx.x == 0 && threadIdx.x == 0) atomicAdd(&sort_ctl[4], 1u);
    __syncthreads();
    // keys of similar magnitude share their high digits, so lanes with equal digits add once
    const unsigned long long stride = (unsigned long long)gridDim.x * blockDim.x;
    const unsigned long long p0 = (unsigned long long)blockIdx.x * blockDim.x + threadIdx.x;
    const unsigned long long rounds = (size + stride - 1) / stride;
    const int lane = threadIdx.x & 31;
    for (unsigned long long r = 0; r < rounds; ++r) {
        const unsigned long long p = p0 + r * stride;
        const bool ok = p < size;
        const unsigned k = ok ? key_of_raw(raw[p]) : 0u;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const unsigned dg = ok ? (k >> (8 * b)) & 255u : 256u;
            const unsigned peers = __match_any_sync(kFull, dg);
            if (ok && (__ffs(peers) - 1) == lane) atomicAdd(&s_h[256 * b + dg], (unsigned)__popc(peers));
        }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < 4 * 256; i += blockDim.x)
        if (s_h[i]) atomicAdd(&digit_hist[i], s_h[i]);
}

constexpr unsigned long long kFlagAgg = 1ull, kFlagInc = 2ull;
constexpr int kSpinLimit = 1 << 20;  // look-back polls before the wait is declared lost

__device__ __forceinline__ unsigned long long status_word(unsigned epoch, unsigned long long flag,
                                                          unsigned count)
{
    return ((unsigned long long)(epoch & 0x3FFFFFFFu) << 34) | (flag << 32) | count;
}

// One pass of the sort (8 bits at `shift`), one kernel.  Tiles take their index in start
// order, so every predecessor of a tile is already running.  A tile ranks its keys stably
// (per-warp running counts; lanes with equal digits found by bit ballots), publishes its digit
// counts, and learns how many keys of each digit precede it from two levels of published
// words: the totals of the earlier groups of 16 tiles (each published by the group's last tile)
// and the counts of the earlier tiles of its own group -- one round of loads, no chain.  The
// digit's global start comes from the pass histogram.  The tile is then staged in digit order
// in shared memory and every digit's run is written contiguously.
__global__ void __launch_bounds__(kThreads) k_rs_onesweep(const float *raw, const unsigned *keys_in,
                                                           const unsigned *vals_in, unsigned *keys_out,
                                                           unsigned *vals_out, unsigned long long size,
                                                           int pass, unsigned ntiles, unsigned *digit_hist,
                                                           unsigned long long *status, unsigned *sort_ctl,
                                                           unsigned *err)
{
    __shared__ unsigned s_base[256];
    __shared__ unsigned s_toff[256], s_gstart[256];
    __shared__ unsigned s_wcnt[kWarps][256];
    __shared__ unsigned s_keys[kTile], s_vals[kTile];
    __shared__ unsigned s_tile, s_epoch;
    __shared__ unsigned s_warp_tot[kWarps];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int shift = 8 * pass;
    const unsigned ngroups = (ntiles + kGroup - 1) / kGroup;
    for (int w = 0; w < kWarps; ++w) s_wcnt[w][tid] = 0;
    pdl_wait();
    pdl_release();
    // the digit's global start: exclusive scan of this pass's histogram
    const unsigned c = digit_hist[pass * 256 + tid];
    unsigned incl = c;
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned v = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) s_warp_tot[warp] = incl;
    __syncthreads();
    unsigned before = 0;
    for (int w = 0; w < warp; ++w) before += s_warp_tot[w];
    s_base[tid] = before + incl - c;
    if (tid == 0) {
        s_epoch = sort_ctl[4];
        s_tile = atomicAdd(&sort_ctl[pass], 1u);
    }
    __syncthreads();
    const unsigned tile = s_tile, epoch = s_epoch;
    if (tile == ntiles - 1) {
        // every tile index has been handed out, so every tile has read the histogram row
        digit_hist[pass * 256 + tid] = 0;
        if (tid == 0) sort_ctl[pass] = 0;
    }

    // local stable ranking: warp w takes keys [tile*4096 + w*512, +512) in 16 rounds of 32
    const unsigned long long base = (unsigned long long)tile * kTile + (unsigned long long)warp * (kTile / kWarps);
    unsigned k[kItems], v[kItems], rk[kItems];
    const unsigned lt = (1u << lane) - 1u;
    // every key and value of the thread first, in one round of loads (the ranking loop below
    // synchronises the warp, which loads may not cross)
#pragma unroll
    for (int i = 0; i < kItems; ++i) {
        const unsigned long long p = base + (unsigned long long)i * 32 + lane;
        const bool ok = p < size;
        k[i] = ok ? (raw ? key_of_raw(__ldg(raw + p)) : __ldg(keys_in + p)) : 0u;
        v[i] = ok ? (raw ? (unsigned)p : __ldg(vals_in + p)) : 0u;
    }
#pragma unroll
    for (int i = 0; i < kItems; ++i) {
        const unsigned long long p = base + (unsigned long long)i * 32 + lane;
        const bool ok = p < size;
        const unsigned dg = ok ? (k[i] >> shift) & 255u : 256u;
        // lanes with this lane's digit: one ballot per digit bit (and one for validity)
        unsigned peers = __ballot_sync(kFull, ok);
        if (!ok) peers = ~peers;
#pragma unroll
        for (int b = 0; b < 8; ++b) {
            const unsigned bit = (dg >> b) & 1u;
            const unsigned bb = __ballot_sync(kFull, bit);
            peers &= bit ? bb : ~bb;
        }
        const unsigned bef = __popc(peers & lt);
        rk[i] = ok ? s_wcnt[warp][dg] + bef : 0;
        __syncwarp();
        if (ok && bef == 0) s_wcnt[warp][dg] += __popc(peers);
        __syncwarp();
    }
    __syncthreads();
    // this tile's count of digit tid, the start of its run within the tile, and the tile
    // staged in digit order in shared memory (which frees the key registers for the look-back)
    unsigned cnt = 0;
    for (int w = 0; w < kWarps; ++w) cnt += s_wcnt[w][tid];
    {
        unsigned inc = cnt;
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned x = __shfl_up_sync(kFull, inc, o);
            if (lane >= o) inc += x;
        }
        if (lane == 31) s_warp_tot[warp] = inc;
        __syncthreads();
        unsigned bef = 0;
        for (int w = 0; w < warp; ++w) bef += s_warp_tot[w];
        s_toff[tid] = bef + inc - cnt;
        unsigned run = bef + inc - cnt;   // per warp, within the tile
        for (int w = 0; w < kWarps; ++w) {
            const unsigned cw = s_wcnt[w][tid];
            s_wcnt[w][tid] = run;
            run += cw;
        }
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < kItems; ++i) {
        const unsigned long long p = base + (unsigned long long)i * 32 + lane;
        if (p < size) {
            const unsigned dg = (k[i] >> shift) & 255u;
            const unsigned tpos = s_wcnt[warp][dg] + rk[i];
            s_keys[tpos] = k[i];
            s_vals[tpos] = v[i];
        }
    }
    // keys of digit tid in earlier tiles: the totals of the earlier complete groups of
    // kGroup tiles plus the counts of the earlier tiles of this tile's group
    unsigned long long *row = status + ((unsigned long long)pass * ntiles) * 256;
    unsigned long long *grow = status + 4ull * ntiles * 256 + (unsigned long long)pass * ngroups * 256;
    volatile unsigned long long *vrow = row, *vgrow = grow;
    const unsigned want = epoch & 0x3FFFFFFFu;
    vrow[(unsigned long long)tile * 256 + tid] = status_word(epoch, kFlagAgg, cnt);
    const unsigned grp = tile / kGroup, first = grp * kGroup;
    bool lost = false;
    if (tile % kGroup == kGroup - 1) {  // the last tile of a group publishes the group total
        unsigned gsum = cnt;
        unsigned long long wv[kGroup - 1];
#pragma unroll
        for (int q = 0; q < kGroup - 1; ++q) wv[q] = vrow[(unsigned long long)(first + q) * 256 + tid];
#pragma unroll
        for (int q = 0; q < kGroup - 1; ++q) {
            unsigned long long w = wv[q];
            int it = 0;
            while (!lost && ((unsigned)(w >> 34) != want || ((w >> 32) & 3ull) == 0) && ++it < kSpinLimit)
                w = vrow[(unsigned long long)(first + q) * 256 + tid];
            if (it >= kSpinLimit) lost = true;
            gsum += (unsigned)w;
        }
        vgrow[(unsigned long long)grp * 256 + tid] = status_word(epoch, kFlagAgg, gsum);
    }
    unsigned excl = 0;
    {
        unsigned long long tv[kGroup - 1];
#pragma unroll
        for (int q = 0; q < kGroup - 1; ++q)
            tv[q] = first + q < tile ? vrow[(unsigned long long)(first + q) * 256 + tid] : 0ull;
        // group totals, kMaxGroups per round (one round up to 2^20 keys)
        for (unsigned q0 = 0; q0 < grp; q0 += kMaxGroups) {
            unsigned long long gv[kMaxGroups];
#pragma unroll
            for (int q = 0; q < kMaxGroups; ++q)
                gv[q] = q0 + q < grp ? vgrow[(unsigned long long)(q0 + q) * 256 + tid] : 0ull;
#pragma unroll
            for (int q = 0; q < kMaxGroups; ++q) {
                if (q0 + q >= grp) continue;
                unsigned long long w = gv[q];
                int it = 0;
                while (!lost && ((unsigned)(w >> 34) != want || ((w >> 32) & 3ull) == 0) && ++it < kSpinLimit)
                    w = vgrow[(unsigned long long)(q0 + q) * 256 + tid];
                if (it >= kSpinLimit) lost = true;
                excl += (unsigned)w;
            }
        }
#pragma unroll
        for (int q = 0; q < kGroup - 1; ++q) {
            if (first + q >= tile) continue;
            unsigned long long w = tv[q];
            int it = 0;
            while (!lost && ((unsigned)(w >> 34) != want || ((w >> 32) & 3ull) == 0) && ++it < kSpinLimit)
                w = vrow[(unsigned long long)(first + q) * 256 + tid];
            if (it >= kSpinLimit) lost = true;
            excl += (unsigned)w;
        }
    }
    if (lost) atomicOr(err, kFlagTimeout);  // a wait gave up: this sort's output is not valid
    s_gstart[tid] = s_base[tid] + excl;
    __syncthreads();
    const unsigned long long tbase = (unsigned long long)tile * kTile;
    const int nvalid = size - tbase < (unsigned long long)kTile ? (int)(size - tbase) : kTile;
    for (int t = tid; t < nvalid; t += blockDim.x) {
        const unsigned key = s_keys[t];
        const unsigned dg = (key >> shift) & 255u;
        const unsigned pos = s_gstart[dg] + (unsigned)t - s_toff[dg];
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

}  // namespace

cudaError_t init_rank_kernels(int carveout)
{
    if (carveout < 0) return cudaSuccess;
    const void *fns[] = {(const void *)k_rs_hist4, (const void *)k_rs_onesweep, (const void *)k_build_cdf};
    for (const void *f : fns) {
        const cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributePreferredSharedMemoryCarveout, carveout);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
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

cudaError_t launch_rank_sort(RankWork &w, unsigned long long host_size, unsigned **sorted, cudaStream_t st)
{
    const unsigned long long size = host_size;
    const unsigned ntiles = (unsigned)std::max<unsigned long long>(rank_tile_count(size), 1);
    const unsigned hgrid = (unsigned)std::min<unsigned long long>((size + kThreads * 16ull - 1) / (kThreads * 16ull), 512);
    cudaError_t e = launch_pdl(k_rs_hist4, std::max(hgrid, 1u), kThreads, 0, st, (const float *)w.raw, size,
                               w.digit_hist, w.sort_ctl);
    if (e != cudaSuccess) return e;
    const unsigned *kin = nullptr, *vin = nullptr;
    int cur = 0;
    for (int pass = 0; pass < 4; ++pass) {
        const float *raw = pass == 0 ? w.raw : nullptr;
        unsigned *kout = pass == 3 ? nullptr : w.keys[cur];
        unsigned *vout = w.vals[cur];
        e = launch_pdl(k_rs_onesweep, ntiles, kThreads, 0, st, raw, kin, vin, kout, vout, size, pass, ntiles,
                       w.digit_hist, (unsigned long long *)w.status, w.sort_ctl, w.err);
        if (e != cudaSuccess) return e;
        kin = w.keys[cur];
        vin = w.vals[cur];
        cur ^= 1;
    }
    *sorted = const_cast<unsigned *>(vin);
    return cudaSuccess;
}

}  // namespace gbper

// ------------------------------------------------------------------------------------------
// per_rank_order_noalloc: the same descending sort for callers that may not allocate device
// memory.  Its scratch (key and value ping-pong buffers, tile histograms) is a file-scope
// device array of fixed size, resolved to a device address once per device.
// ------------------------------------------------------------------------------------------
#include "gbper.h"

#include <mutex>

namespace gbper {
namespace {

constexpr unsigned long long kNoAllocMaxKeys = 1ull << 18;
constexpr unsigned long long kNoAllocTiles = (kNoAllocMaxKeys + kTile - 1) / kTile;
constexpr unsigned long long kNoAllocGroups = (kNoAllocTiles + kGroup - 1) / kGroup;
// keys[2], values[2], digit histograms, sort control, then 64-bit look-back words
constexpr unsigned long long kNoAllocWords =
    4 * kNoAllocMaxKeys + 1024 + 16 + 2 * (4 * (kNoAllocTiles + kNoAllocGroups) * 256);
constexpr int kNoAllocMaxDevices = 64;

// About 4.5 MiB per device, held by every device that loads the library until exit;
// zero at load, which the sort's histograms, control words and epoch tags rely on.
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

}  // namespace

}  // namespace gbper

extern "C" per_status per_rank_order_noalloc(const float *d_raw, uint32_t n, uint32_t *d_order,
                                             void *stream)
{
    using namespace gbper;
    if (!d_raw || !d_order || n == 0 || n > kNoAllocMaxKeys) return PER_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(d_raw) % 4 || reinterpret_cast<uintptr_t>(d_order) % 4)
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
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    unsigned *sorted = nullptr;
    cudaError_t e = launch_rank_sort(w, n, &sorted, st);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(d_order, sorted, (size_t)n * sizeof(unsigned), cudaMemcpyDeviceToDevice, st);
    return e == cudaSuccess ? PER_OK : PER_ERR_CUDA;
}
