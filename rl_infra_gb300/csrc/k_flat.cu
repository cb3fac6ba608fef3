// k_flat.cu -- the cumulative array of flat mode ("GPU-Resident Prioritized Experience Replay",
// Sampling Kernels, Proportional step 2: an inclusive sum of the priorities, searched per draw).
//
// The sums run on the integer pipe in fixed point (GB300's binary64 pipe retires a warp
// instruction only every few dozen cycles per SM; its integer pipes retire several per cycle).
// With E the biased exponent of the running maximum leaf, the unit is 2^(E - 178): the largest
// leaf is below 2^52 units and keeps every bit; a smaller leaf is rounded to the unit (to
// nearest), an error of at most 2^-53 of the largest leaf's binade, as for one binary64 add.  A
// 2048-leaf tile's sums fit in 64 bits; the sums of the tiles before a tile are kept in 128 bits.
// Integer sums do not depend on their order, so each C[i] is the fixed-point prefix rounded once
// to binary64 (to nearest, ties to even): its error against the exact sum of the leaves is at
// most half a unit per slot plus that one rounding, on the order of binary64's own summation.
//   k_flat_reduce  one 2048-leaf tile per CTA (8 per thread): the tile's sum and minimum; the
//                  last CTA to arrive turns the tile sums into the sums of the tiles before each.
//   k_flat_scan    the same tiles again: prefix sums inside the tile (registers, warp shuffles,
//                  the warps' totals) plus the tile's offset, rounded and stored as C; the thread
//                  holding slot size-1 records T = C[size-1].
// No CTA waits for another.
#include "per_internal.cuh"

namespace gbper {

namespace {

constexpr int kThreads = 256;
constexpr int kPer = 8;
constexpr int kTile = kThreads * kPer;
constexpr float kInf = __builtin_huge_valf();
constexpr int kUnitBias = 178;   // unit = 2^(E - kUnitBias)

typedef unsigned __int128 u128;

// A leaf in units of 2^(emax - 178), rounded to nearest: its 24-bit significand shifted by
// e - emax + 28.  Leaves never exceed the running maximum leaf (e <= emax); capped anyway.
__device__ __forceinline__ unsigned long long leaf_fixed(float f, int emax)
{
    const unsigned b = __float_as_uint(f);
    if (b == 0u) return 0ull;
    const int e = (int)(b >> 23);
    const unsigned long long m = e ? (unsigned long long)((b & 0x7fffffu) | 0x800000u) : (unsigned long long)b;
    int s = (e ? e : 1) - emax + 28;
    if (s > 28) s = 28;
    if (s >= 0) return m << s;
    if (s < -25) return 0ull;
    return (m + (1ull << (-s - 1))) >> (-s);
}

// (hi, lo) units (a 128-bit integer) rounded to binary64, to nearest, ties to even
__device__ __forceinline__ double fixed_to_double(unsigned long long hi, unsigned long long lo, int emax)
{
    int p;
    unsigned long long top;   // the 64 bits from the leading one down
    bool sticky;              // any bit below them
    if (hi != 0ull) {
        const int lz = __clzll((long long)hi);
        p = 127 - lz;
        top = lz ? (hi << lz) | (lo >> (64 - lz)) : hi;
        sticky = (lz ? (lo << lz) : lo) != 0ull;
    } else {
        if (lo == 0ull) return 0.0;
        const int lz = __clzll((long long)lo);
        p = 63 - lz;
        top = lo << lz;
        sticky = false;
    }
    unsigned long long mant = top >> 11;
    const unsigned long long rem = top & 0x7ffull;
    if (rem > 0x400ull || (rem == 0x400ull && (sticky || (mant & 1ull)))) {
        mant += 1ull;
        if (mant == (1ull << 53)) {
            mant >>= 1;
            p += 1;
        }
    }
    const long long e = (long long)p + (emax - kUnitBias) + 1023;
    return __longlong_as_double((long long)(((unsigned long long)e << 52) | (mant & ((1ull << 52) - 1ull))));
}

// This thread's 8 leaves (0 past the filled slots).
__device__ __forceinline__ void load_leaves(const float *L, unsigned long long i0, unsigned long long size,
                                            float *lf)
{
    if (i0 + kPer <= size) {
        const float4 x = reinterpret_cast<const float4 *>(L + i0)[0];
        const float4 y = reinterpret_cast<const float4 *>(L + i0)[1];
        lf[0] = x.x; lf[1] = x.y; lf[2] = x.z; lf[3] = x.w;
        lf[4] = y.x; lf[5] = y.y; lf[6] = y.z; lf[7] = y.w;
    } else {
#pragma unroll
        for (int k = 0; k < kPer; ++k) lf[k] = i0 + k < size ? L[i0 + k] : 0.0f;
    }
}

__device__ __forceinline__ bool last_cta_to_arrive(unsigned *ticket)
{
    __shared__ int s_last;
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = atomicAdd(ticket, 1u) == gridDim.x - 1;
    __syncthreads();
    if (s_last) __threadfence();
    return s_last != 0;
}

// Exclusive prefix of one value per thread across the CTA; returns it and the CTA's total.
__device__ __forceinline__ unsigned long long block_exclusive(unsigned long long v, unsigned long long *total)
{
    __shared__ unsigned long long s_w[kThreads / 32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    unsigned long long inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long y = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += y;
    }
    if (lane == 31) s_w[warp] = inc;
    __syncthreads();
    unsigned long long before = 0ull, all = 0ull;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) {
        const unsigned long long t = s_w[w];
        if (w < warp) before += t;
        all += t;
    }
    __syncthreads();
    *total = all;
    return before + inc - v;
}

__global__ void __launch_bounds__(kThreads) k_flat_reduce(const float *L, FlatWork fw, Ctl *ctl)
{
    __shared__ float s_mn[kThreads / 32];
    pdl_wait();
    pdl_release();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const unsigned long long size = ctl->size;
    const int emax = (int)(ctl->max_leaf_bits >> 23);
    const unsigned long long t0 = (unsigned long long)blockIdx.x * kTile;
    if (t0 < size) {
        float lf[kPer];
        const unsigned long long i0 = t0 + (unsigned long long)kPer * tid;
        load_leaves(L, i0, size, lf);
        unsigned long long sum = 0ull;
        float mn = kInf;
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
            sum += leaf_fixed(lf[k], emax);
            if (i0 + k < size) mn = fminf(mn, lf[k]);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
        if (lane == 0) s_mn[warp] = mn;
        unsigned long long total;
        block_exclusive(sum, &total);
        if (tid == 0) {
            float m = kInf;
#pragma unroll
            for (int w = 0; w < kThreads / 32; ++w) m = fminf(m, s_mn[w]);
            fw.agg[blockIdx.x] = total;
            fw.tmin[blockIdx.x] = m;
        }
    }
    if (!last_cta_to_arrive(fw.tick)) return;
    // the sums of the tiles before each active tile (thread t takes a contiguous run of tiles),
    // and the smallest filled leaf
    const unsigned long long nt = (size + kTile - 1) / kTile;
    const unsigned long long per = (nt + kThreads - 1) / kThreads;
    const unsigned long long a = (unsigned long long)tid * per < nt ? (unsigned long long)tid * per : nt;
    const unsigned long long b = a + per < nt ? a + per : nt;
    u128 own = 0;
    float m = kInf;
    for (unsigned long long t = a; t < b; ++t) {
        own += __ldcg(fw.agg + t);
        m = fminf(m, __ldcg(fw.tmin + t));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fminf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) s_mn[warp] = m;
    // exclusive prefix of the 256 runs' 128-bit sums
    __shared__ unsigned long long s_lo[kThreads], s_hi[kThreads];
    s_lo[tid] = (unsigned long long)own;
    s_hi[tid] = (unsigned long long)(own >> 64);
    __syncthreads();
    for (int o = 1; o < kThreads; o <<= 1) {
        u128 v = ((u128)s_hi[tid] << 64) | s_lo[tid];
        if (tid >= o) v += ((u128)s_hi[tid - o] << 64) | s_lo[tid - o];
        __syncthreads();
        s_lo[tid] = (unsigned long long)v;
        s_hi[tid] = (unsigned long long)(v >> 64);
        __syncthreads();
    }
    u128 run = ((u128)s_hi[tid] << 64 | s_lo[tid]) - own;
    for (unsigned long long t = a; t < b; ++t) {
        const unsigned long long v = __ldcg(fw.agg + t);
        fw.excl[2 * t] = (unsigned long long)run;
        fw.excl[2 * t + 1] = (unsigned long long)(run >> 64);
        run += v;
    }
    if (tid == 0) {
        float mm = kInf;
#pragma unroll
        for (int w = 0; w < kThreads / 32; ++w) mm = fminf(mm, s_mn[w]);
        fw.res[2] = __float_as_uint(mm);
        fw.tick[0] = 0u;
    }
}

__global__ void __launch_bounds__(kThreads) k_flat_scan(const float *L, FlatWork fw, Ctl *ctl)
{
    pdl_wait();
    pdl_release();
    const int tid = threadIdx.x;
    const unsigned long long size = ctl->size;
    const int emax = (int)(ctl->max_leaf_bits >> 23);
    const unsigned long long t0 = (unsigned long long)blockIdx.x * kTile;
    if (t0 >= size) return;
    float lf[kPer];
    const unsigned long long i0 = t0 + (unsigned long long)kPer * tid;
    load_leaves(L, i0, size, lf);
    const u128 off = ((u128)__ldcg(fw.excl + 2ull * blockIdx.x + 1) << 64) | __ldcg(fw.excl + 2ull * blockIdx.x);
    unsigned long long p[kPer];
    unsigned long long acc = 0ull;
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
        acc += leaf_fixed(lf[k], emax);
        p[k] = acc;
    }
    unsigned long long total;
    const u128 base = off + block_exclusive(acc, &total);
    double c[kPer];
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
        const u128 x = base + p[k];
        c[k] = fixed_to_double((unsigned long long)(x >> 64), (unsigned long long)x, emax);
    }
    if (i0 + kPer <= size) {
        double2 *dst = reinterpret_cast<double2 *>(fw.C + i0);
#pragma unroll
        for (int k = 0; k < kPer; k += 2) dst[k / 2] = make_double2(c[k], c[k + 1]);
    } else {
#pragma unroll
        for (int k = 0; k < kPer; ++k)
            if (i0 + k < size) fw.C[i0 + k] = c[k];
    }
#pragma unroll
    for (int k = 0; k < kPer; ++k)
        if (i0 + k + 1 == size) fw.res[1] = (unsigned long long)__double_as_longlong(c[k]);
}

}  // namespace

unsigned long long flat_tiles(unsigned long long capacity) { return (capacity + kTile - 1) / kTile; }

cudaError_t launch_flat_scan(const float *L, const FlatWork &fw, Ctl *ctl, unsigned long long capacity,
                             cudaStream_t st)
{
    const unsigned grid = (unsigned)flat_tiles(capacity);
    cudaError_t e = launch_pdl(k_flat_reduce, grid, kThreads, 0, st, L, fw, ctl);
    if (e == cudaSuccess) e = launch_pdl(k_flat_scan, grid, kThreads, 0, st, L, fw, ctl);
    return e;
}

}  // namespace gbper
