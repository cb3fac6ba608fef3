// k_rank.cu -- rank-based prioritization: the stable descending sort of (raw priority, slot)
// and the rank CDF ("GPU-Resident Prioritized Experience Replay", Sampling Kernels,
// Rank-based: sort (priority, index) pairs descending, then probabilities 1/rank^alpha and
// their cumulative sum).
//
// Sort: least-significant-digit radix sort, four passes of 8 bits over the key ~bits(raw)
// (raw > 0, so ascending ~bits is descending raw), values = slot.  Each pass is
// reduce-then-scan with no inter-CTA waiting:
//   tile_hist  per 4096-key tile, a 256-bin histogram, stored digit-major [256][tiles];
//   scan       one exclusive scan of that digit-major array gives, for every (digit, tile),
//              where the tile's keys of that digit start in the output;
//   scatter    each tile ranks its keys stably (warp match + per-warp running counts) and
//              writes them to their final positions.
// Pass 0 reads the raw priorities directly and makes the slot values on the fly; the last
// pass writes only the slot values.  Ties keep ascending slot order because every pass is
// stable and pass 0 starts in slot order.
#include "per_internal.cuh"

#include <algorithm>

namespace gbper {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kItems = 16;                       // keys per thread per tile
constexpr int kTile = kThreads * kItems;          // 4096
constexpr int kScanThreads = 1024;
constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ unsigned key_of_raw(float raw) { return ~__float_as_uint(raw); }

__global__ void __launch_bounds__(kThreads) k_rs_tile_hist(const float *raw, const unsigned *keys,
                                                            unsigned long long size, int shift,
                                                            unsigned *tile_hist, unsigned ntiles)
{
    __shared__ unsigned s_hist[256];
    s_hist[threadIdx.x] = 0;
    __syncthreads();
    const unsigned long long base = (unsigned long long)blockIdx.x * kTile;
#pragma unroll
    for (int i = 0; i < kItems; ++i) {
        const unsigned long long p = base + (unsigned long long)i * kThreads + threadIdx.x;
        if (p < size) {
            const unsigned k = raw ? key_of_raw(raw[p]) : keys[p];
            atomicAdd(&s_hist[(k >> shift) & 255u], 1u);
        }
    }
    __syncthreads();
    tile_hist[(unsigned long long)threadIdx.x * ntiles + blockIdx.x] = s_hist[threadIdx.x];
}

// Exclusive scan of tile_hist[0, count) in place, one CTA.
__global__ void __launch_bounds__(kScanThreads) k_rs_scan(unsigned *h, unsigned long long count)
{
    __shared__ unsigned s_warp[kScanThreads / 32];
    const unsigned long long per = (count + kScanThreads - 1) / kScanThreads;
    const unsigned long long beg = threadIdx.x * per;
    unsigned sum = 0;
    for (unsigned long long i = 0; i < per; ++i)
        if (beg + i < count) sum += h[beg + i];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    unsigned incl = sum;
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned v = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        unsigned v = s_warp[lane];
        unsigned inc = v;
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned x = __shfl_up_sync(kFull, inc, o);
            if (lane >= o) inc += x;
        }
        s_warp[lane] = inc - v;
    }
    __syncthreads();
    unsigned run = s_warp[warp] + incl - sum;
    for (unsigned long long i = 0; i < per; ++i)
        if (beg + i < count) {
            const unsigned v = h[beg + i];
            h[beg + i] = run;
            run += v;
        }
}

__global__ void __launch_bounds__(kThreads) k_rs_scatter(const float *raw, const unsigned *keys_in,
                                                          const unsigned *vals_in, unsigned *keys_out,
                                                          unsigned *vals_out, unsigned long long size,
                                                          int shift, const unsigned *tile_off,
                                                          unsigned ntiles)
{
    __shared__ unsigned s_off[256];
    __shared__ unsigned s_wcnt[kWarps][256];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    s_off[tid] = tile_off[(unsigned long long)tid * ntiles + blockIdx.x];
    for (int w = 0; w < kWarps; ++w) s_wcnt[w][tid] = 0;
    __syncthreads();
    const unsigned long long base = (unsigned long long)blockIdx.x * kTile + (unsigned long long)warp * (kTile / kWarps);
    unsigned k[kItems], v[kItems], rk[kItems];
    const unsigned lt = (1u << lane) - 1u;
#pragma unroll
    for (int i = 0; i < kItems; ++i) {
        const unsigned long long p = base + (unsigned long long)i * 32 + lane;
        const bool ok = p < size;
        if (ok) {
            k[i] = raw ? key_of_raw(raw[p]) : keys_in[p];
            v[i] = raw ? (unsigned)p : vals_in[p];
        } else {
            k[i] = 0;
            v[i] = 0;
        }
        const unsigned dg = ok ? (k[i] >> shift) & 255u : 256u;
        const unsigned peers = __match_any_sync(kFull, dg);
        const unsigned before = __popc(peers & lt);
        rk[i] = ok ? s_wcnt[warp][dg] + before : 0;
        __syncwarp();
        if (ok && before == 0) s_wcnt[warp][dg] += __popc(peers);
        __syncwarp();
    }
    __syncthreads();
    {   // per digit: exclusive scan over the warps, plus the tile's global start
        unsigned run = s_off[tid];
        for (int w = 0; w < kWarps; ++w) {
            const unsigned c = s_wcnt[w][tid];
            s_wcnt[w][tid] = run;
            run += c;
        }
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < kItems; ++i) {
        const unsigned long long p = base + (unsigned long long)i * 32 + lane;
        if (p < size) {
            const unsigned dg = (k[i] >> shift) & 255u;
            const unsigned pos = s_wcnt[warp][dg] + rk[i];
            if (keys_out) keys_out[pos] = k[i];
            vals_out[pos] = v[i];
        }
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
    const void *fns[] = {(const void *)k_rs_tile_hist, (const void *)k_rs_scan, (const void *)k_rs_scatter,
                         (const void *)k_build_cdf};
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

cudaError_t launch_rank_sort(RankWork &w, unsigned long long host_size, unsigned **sorted, cudaStream_t st)
{
    const unsigned long long size = host_size;
    const unsigned ntiles = (unsigned)std::max<unsigned long long>(rank_tile_count(size), 1);
    const unsigned *kin = nullptr, *vin = nullptr;
    int cur = 0;
    for (int pass = 0; pass < 4; ++pass) {
        const int shift = 8 * pass;
        const float *raw = pass == 0 ? w.raw : nullptr;
        k_rs_tile_hist<<<ntiles, kThreads, 0, st>>>(raw, kin, size, shift, w.tile_hist, ntiles);
        k_rs_scan<<<1, kScanThreads, 0, st>>>(w.tile_hist, 256ull * ntiles);
        unsigned *kout = pass == 3 ? nullptr : w.keys[cur];
        unsigned *vout = w.vals[cur];
        k_rs_scatter<<<ntiles, kThreads, 0, st>>>(raw, kin, vin, kout, vout, size, shift, w.tile_hist, ntiles);
        const cudaError_t e = cudaGetLastError();
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
constexpr unsigned long long kNoAllocWords = 4 * kNoAllocMaxKeys + 256 * kNoAllocTiles;
constexpr int kNoAllocMaxDevices = 64;

// 4 MiB + 64 KiB per device, held by every device that loads the library until exit.
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
    w.tile_hist = base + 4 * kNoAllocMaxKeys;
    w.capacity = n;
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    unsigned *sorted = nullptr;
    cudaError_t e = launch_rank_sort(w, n, &sorted, st);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(d_order, sorted, (size_t)n * sizeof(unsigned), cudaMemcpyDeviceToDevice, st);
    return e == cudaSuccess ? PER_OK : PER_ERR_CUDA;
}
