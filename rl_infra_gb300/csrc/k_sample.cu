// k_sample.cu -- stratified sampling, importance weights and the row gather, fused.
//
// Proportional mode ("GPU-Resident Prioritized Experience Replay", Sampling Kernels,
// Proportional; "Putting prioritized replay's segment tree on a GPU", Sampling Is a Descent).
// One warp serves one draw j:
//   u_j     Philox4x32-10, counter (j, call, tag 0)
//   mass_j  (j + u_j) * (T / B): one draw per stratum of [0, T)
//   descent the same walk as the post's st_find_prefixsum_idx (left when the left child's sum
//           exceeds the mass, otherwise subtract and go right), evaluated in an order that
//           reaches the same decisions with few dependent memory round trips: the warp loads
//           the 2^k - 1 left children of a k-level subtree (k <= 7) in one round, four per
//           lane, and walks those k levels with shuffles; the last round loads the leaves under
//           its node as one contiguous stretch.  A 2^21-leaf tree takes three rounds.  Every
//           comparison and subtraction is the binary64 operation of the sequential walk (the
//           compare on the integer pipe, since the operands are non-negative), so the leaf and
//           the leftover mass are bit-identical to it.
//   weight  w = (n P(i))^-beta / max_w with max_w from the min tree, i.e. (L[i]/p_min)^-beta
//   gather  the warp copies the chosen rows (zero-padded to the output stride, as the padded
//           gather of "True Single-Graph Implementation Plan", Task 2) and the scalars.
// Each CTA takes the call number from the device-side counter when it starts; the last to
// start advances it.
#include "per_internal.cuh"

#include <algorithm>
#include <cstdlib>

namespace gbper {

namespace {

constexpr int kThreads = 256;
constexpr unsigned kFull = 0xffffffffu;

struct SampleArgs {
    TreeRefs t;
    RingRefs r;
    Ctl *ctl;
    unsigned B;
    double inv_b;   // 1/B when B is a power of two (exact), else 0
    float beta;
    unsigned long long seed;
    SampleOut o;
    int vec4;  // rows move as float4
    int top;   // levels walked from the copy of the tree's top in shared memory (0: none)
};

// The sampled row, copied by the G lanes that served the draw: every load of a chunk of G V
// float4 of the row pair (and the action, reward and done fields on lanes 1-3) is issued before
// the chunk's first store, so the gather costs one memory round trip per chunk (one for rows of up
// to 256 floats with G V = 128).  Rows shorter than the output stride are padded with zeros.
template <int G, int V>
__device__ __forceinline__ void gather_row(const RingRefs &r, const SampleOut &o, unsigned j,
                                           unsigned long long slot, int lane, int vec4)
{
    const unsigned d = r.d, dp = o.dp;
    unsigned act = 0;
    float rew = 0.0f;
    unsigned char done = 0;
    if (lane == 1 && o.actions) act = __ldg(r.actions + slot);
    if (lane == 2 && o.rewards) rew = __ldg(r.rewards + slot);
    if (lane == 3 && o.dones) done = __ldg(r.dones + slot);
    const bool rows = dp && (o.states || o.next);   // with d = 0 the rows are all padding
    if (rows && vec4) {
        // the row pair as 2 dp4 float4, in chunks of G V: V per lane, all loaded before any store
        const unsigned d4 = d >> 2, dp4 = dp >> 2;
        const float4 *srcS = reinterpret_cast<const float4 *>(r.states + slot * d);
        const float4 *srcN = reinterpret_cast<const float4 *>(r.next + slot * d);
        const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
        for (unsigned c0 = 0; c0 < 2 * dp4; c0 += G * V) {
            float4 v[V];
#pragma unroll
            for (int q = 0; q < V; ++q) {
                const unsigned c = c0 + lane + G * q;
                const bool second = c >= dp4;
                const unsigned cc = second ? c - dp4 : c;
                v[q] = zero;
                if (c < 2 * dp4 && cc < d4 && (second ? o.next : o.states)) v[q] = __ldg((second ? srcN : srcS) + cc);
            }
#pragma unroll
            for (int q = 0; q < V; ++q) {
                const unsigned c = c0 + lane + G * q;
                const bool second = c >= dp4;
                const unsigned cc = second ? c - dp4 : c;
                float *base = second ? o.next : o.states;
                if (c < 2 * dp4 && base) reinterpret_cast<float4 *>(base + (unsigned long long)j * dp)[cc] = v[q];
            }
        }
    } else if (rows) {
        for (unsigned c = lane; c < 2 * dp; c += G) {
            const bool second = c >= dp;
            const unsigned cc = second ? c - dp : c;
            float *dst = second ? o.next : o.states;
            if (!dst) continue;
            const float *src = second ? r.next : r.states;
            dst[(unsigned long long)j * dp + cc] = cc < d ? __ldg(src + slot * d + cc) : 0.0f;
        }
    }
    if (lane == 1 && o.actions) o.actions[j] = act;
    if (lane == 2 && o.rewards) o.rewards[j] = rew;
    if (lane == 3 && o.dones) {
        if (o.dones_f32) reinterpret_cast<float *>(o.dones)[j] = done ? 1.0f : 0.0f;
        else o.dones[j] = done;
    }
}

// a > b for binary64 values >= +0: their bit patterns order like the values, so the compare
// runs on the integer pipe (GB300's binary64 pipe retires far fewer lanes per cycle).
__device__ __forceinline__ bool gt_nonneg(double a, double b)
{
    return __double_as_longlong(a) > __double_as_longlong(b);
}

// One round of the walk: k levels below `node`, served by G lanes holding S slots each, so
// k <= log2(G S + 1).  The 2^k - 1 left children the walk may read are loaded at once (child i of
// the round sits in lane i % G, slot i / G), and the k decisions then run on registers and
// shuffles within the G lanes.  When `last`, the deepest level is the leaves: the 2^k leaves
// under `node` are one contiguous stretch, S per lane, and *lv receives the chosen leaf's value.
// The loads (walk_load) and the decisions (walk_decide) are separate so that the first round's
// loads, which do not depend on the draw, can be issued before the call number is known.
template <int S>
struct WalkRegs {
    double v[S];
    float lf[S];
};

template <int S>
__device__ __forceinline__ float pick_slot(const float (&v)[S], int r)
{
    float x = v[0];
#pragma unroll
    for (int q = 1; q < S; ++q)
        if (r == q) x = v[q];
    return x;
}

template <int G, int S>
__device__ __forceinline__ void walk_load(const TreeRefs &t, unsigned long long node, int k, bool last,
                                          int lane, WalkRegs<S> &w)
{
    const int ninternal = (1 << (last ? k - 1 : k)) - 1;  // left children that are internal nodes
#pragma unroll
    for (int r = 0; r < S; ++r) {
        const int i = lane + G * r;
        w.v[r] = 0.0;
        if (i < ninternal) {
            const int lev = 32 - __clz(i + 1);
            const int pos = i + 1 - (1 << (lev - 1));
            w.v[r] = t.S[(node << lev) + 2 * pos];
        }
        w.lf[r] = 0.0f;
        if (last && i < (1 << k)) w.lf[r] = t.L[(node << k) - t.n + i];
    }
}

// The slot among v[lo .. hi] (lo, hi known once the caller's loop is unrolled): the selects outside
// that range fold away.
template <int S>
__device__ __forceinline__ double pick_slot_in(const double (&v)[S], int r, int lo, int hi)
{
    double x = v[lo];
#pragma unroll
    for (int q = 0; q < S; ++q)
        if (q > lo && q <= hi && r == q) x = v[q];
    return x;
}

template <int G, int S>
__device__ __forceinline__ unsigned long long walk_decide(unsigned long long node, int k, bool last,
                                                          double &m, int lane, const WalkRegs<S> &w,
                                                          float *lv)
{
    int q = 0;
    const int kint = last ? k - 1 : k;
    // unrolled, so that each level picks among the slots its nodes can occupy (children
    // 2^(lev-1) - 1 .. 2^lev - 2 sit in slots i / G); measured on GB300 against a loop at one
    // draw per warp: the apex step 38.5K against 37.7K steps/s, the dqn sample 10.2 against 11.8 us
    constexpr int KM = G * S >= 127 ? 7 : (G * S >= 63 ? 6 : 5);
#pragma unroll
    for (int lev = 1; lev <= KM; ++lev) {
        if (lev <= kint) {
            const int i = (1 << (lev - 1)) - 1 + q;
            const int lo = ((1 << (lev - 1)) - 1) / G, hi = ((1 << lev) - 2) / G;
            const double left = __shfl_sync(kFull, pick_slot_in<S>(w.v, i / G, lo, hi < S ? hi : S - 1),
                                            i & (G - 1), G);
            if (gt_nonneg(left, m)) {
                q = 2 * q;
            } else {
                m = __dsub_rn(m, left);
                q = 2 * q + 1;
            }
        }
    }
    if (last) {
        const int i = 2 * q;  // the left leaf of the final pair
        const double left = (double)__shfl_sync(kFull, pick_slot<S>(w.lf, i / G), i & (G - 1), G);
        if (gt_nonneg(left, m)) {
            q = 2 * q;
        } else {
            m = __dsub_rn(m, left);
            q = 2 * q + 1;
        }
        *lv = __shfl_sync(kFull, pick_slot<S>(w.lf, q / G), q & (G - 1), G);
    }
    return (node << k) + q;
}

// The last round under the shared-memory top reads its leaves only (walk_leaves, up to 4 leaves a
// lane): one line a draw instead of a line for each level of left children.  Deeper rounds of
// internal nodes rebuilt the same way from their bottom rows cut the stress sampler's DRAM reads
// further (8.6 against 11.3 MB a launch with rows of 4 floats) but their pairwise sums cost 10
// more binary64 instructions a warp, about 2 us a stress step on GB300; they stay on left
// children.
constexpr bool kLeafRounds = true;

// The last round of a walk from the 2^k leaves under `node` alone: every stored node is the
// binary64 sum of its two children (the leaves taken as binary64), so the pairwise sums below
// are the k - 1 levels of nodes above the leaves bit for bit.  Lane l of the G holds leaves
// [l R, l R + R), R = 2^LR = 2^k / G: it adds them pairwise in registers, the G lanes add their
// sums pairwise by shuffles, and each of the k decisions takes its left child from the lane
// that holds it.  Returns the leaf's heap index; *lv receives its value.
template <int G, int LR>
__device__ __forceinline__ unsigned long long walk_leaves(const TreeRefs &t, unsigned long long node, double &m,
                                                          int lane, float *lv)
{
    constexpr int LG = G == 32 ? 5 : (G == 16 ? 4 : 3);   // log2(G)
    constexpr int R = 1 << LR;
    const unsigned long long first = node << (LG + LR);   // heap index of the first leaf
    const float *src = t.L + (first - t.n) + (unsigned long long)lane * R;
    float f[R];
    if constexpr (R == 4) {
        const float4 x = *reinterpret_cast<const float4 *>(src);
        f[0] = x.x; f[1] = x.y; f[2] = x.z; f[3] = x.w;
    } else if constexpr (R == 2) {
        const float2 x = *reinterpret_cast<const float2 *>(src);
        f[0] = x.x; f[1] = x.y;
    } else {
        f[0] = src[0];
    }
    // h: the lane's leaves at [0, R), then its pairwise sums level by level (level j at
    // [2R - 2R/2^j, 2R - R/2^j)); the lane's sum at 2R - 2
    double h[2 * R - 1];
#pragma unroll
    for (int r = 0; r < R; ++r) h[r] = (double)f[r];
#pragma unroll
    for (int j = 1; j <= LR; ++j) {
        const int in = 2 * R - (2 * R >> (j - 1)), out = 2 * R - (2 * R >> j);
#pragma unroll
        for (int i = 0; i < (R >> j); ++i) h[out + i] = __dadd_rn(h[in + 2 * i], h[in + 2 * i + 1]);
    }
    // the sums of the lane's blocks of 1, 2, 4, ... lanes: bf[j] covers 2^j lanes
    double bf[LG];
    bf[0] = h[2 * R - 2];
#pragma unroll
    for (int j = 0; j + 1 < LG; ++j) bf[j + 1] = __dadd_rn(bf[j], __shfl_xor_sync(kFull, bf[j], 1 << j, G));
    // levels 1 .. LG choose the lane: the left half of the block of lanes [L, L + 2 half)
    int L = 0;
#pragma unroll
    for (int i = 1; i <= LG; ++i) {
        const double left = __shfl_sync(kFull, bf[LG - i], L, G);
        if (!gt_nonneg(left, m)) {
            m = __dsub_rn(m, left);
            L += G >> i;
        }
    }
    // levels LG + 1 .. k inside lane L: the left child is the first entry of the level just below
    // the current block, and each decision keeps the half of every lower level (and of the
    // leaves) that it took -- selects at fixed positions, so the rows stay in registers
    int q = 0;
#pragma unroll
    for (int i = 1; i <= LR; ++i) {
        const int lvl = LR - i;
        const double left = __shfl_sync(kFull, h[2 * R - (2 * R >> lvl)], L, G);
        const bool right = !gt_nonneg(left, m);
        if (right) {
            m = __dsub_rn(m, left);
            q += R >> i;
        }
#pragma unroll
        for (int j = 0; j < lvl; ++j) {
            const int b = 2 * R - (2 * R >> j), cnt = R >> (j + i);
#pragma unroll
            for (int e = 0; e < cnt; ++e) h[b + e] = right ? h[b + cnt + e] : h[b + e];
        }
#pragma unroll
        for (int e = 0; e < (R >> i); ++e) f[e] = right ? f[(R >> i) + e] : f[e];
    }
    *lv = __shfl_sync(kFull, f[0], L, G);
    return first + (unsigned long long)L * R + q;
}

// G lanes serve one draw (32 / G draws per warp at once), each lane holding S nodes of a round:
// rounds of K = log2(G S + 1) levels (7 for 32 x 4; 6 for 16 x 4 and 8 x 8).  Every level of the
// walk is one binary64 subtraction per warp instruction, and GB300's binary64 pipe retires about
// one warp instruction every 19 cycles per SM, so large batches share each instruction among 2
// or 4 draws; the deepest round also reads 17 sectors of nodes and leaves instead of 33.
// With TOP > 0 (large batches, where every draw walks its own path below the top few levels)
// each CTA copies the nodes of depths 0 .. TOP into shared memory and the first a.top levels of
// every draw are walked there, one node a level; the levels below follow in as few rounds as K
// allows, the shallower rounds taking the extra level (a round of k levels reads about 2^k
// nodes, and below the top every draw reads its own), and the last round reads its leaves alone
// (walk_leaves).  DRAM moves 128-byte lines here: below the levels the draws share, each level
// of left children costs a draw a line, and a round of leaves one line for all its levels.
template <int G, int S, int TOP>
__global__ void __launch_bounds__(kThreads, 2) k_sample_prop(SampleArgs a)
{
    constexpr int K = G * S >= 127 ? 7 : (G * S >= 63 ? 6 : 5);   // levels per round
    constexpr int GV = G >= 16 ? 128 / G : 8;                      // float4 per lane per gather chunk
    constexpr int per_warp = 32 / G;
    constexpr int LG = G == 32 ? 5 : (G == 16 ? 4 : 3);           // log2(G)
    __shared__ unsigned long long s_call;
    __shared__ __align__(16) double s_top[TOP > 0 ? 2 << TOP : 2];
    pdl_wait();
    pdl_release();
    const unsigned long long n = a.t.n;
    const int D = a.t.D;
    if (threadIdx.x == 0) s_call = take_call_number(a.ctl);
    const int top = TOP > 0 ? a.top : 0;   // the host passes 0 or TOP, and TOP < D
    if (TOP > 0 && top > 0) {
        // 16-byte loads, all issued before the first store (the tree's arrays are 256-byte aligned)
        const double2 *src = reinterpret_cast<const double2 *>(a.t.S);
        double2 *dst = reinterpret_cast<double2 *>(s_top);
#pragma unroll 4
        for (int i = threadIdx.x; i < (1 << TOP); i += blockDim.x) dst[i] = src[i];
    }
    // while the call number is on its way: the total, the minimum, the size and the first
    // round's nodes (the same for every draw)
    const double total = D == 0 ? (double)a.t.L[0] : a.t.S[1];
    const float pmin = D == 0 ? leaf_min_value(a.t.L[0]) : a.t.M[1];
    const unsigned long long size = a.ctl->size;
    // rounds below the top: without a top, K levels each and the first takes the rest; with one,
    // kb or kb + 1 levels each, the first kx rounds taking kb + 1
    const int dk = D - top;
    const int rounds = (dk + K - 1) / K;
    const int kb = top > 0 ? dk / rounds : K, kx = top > 0 ? dk % rounds : 0;
    const int first = top > 0 ? kb + (kx != 0) : dk - K * (rounds - 1);
    const int lane = threadIdx.x & (G - 1);
    const unsigned sub = (threadIdx.x & 31) / G;
    // the first round's nodes are preloaded (before the call number arrives) when they fit the
    // register budget beside the gather (one draw per warp); otherwise each draw loads them (L1)
    constexpr bool kPre = G == 32;
    WalkRegs<S> w0;
    if (kPre && D > 0) walk_load<G, S>(a.t, 1, first, rounds == 1, lane, w0);
    // stratum width T / B: one exact scaling when B is a power of two
    const double seg = a.inv_b != 0.0 ? __dmul_rn(total, a.inv_b) : __ddiv_rn(total, (double)a.B);
    __syncthreads();
    const unsigned long long call = s_call;
    const float nbeta = -a.beta;
    const unsigned wpb = blockDim.x >> 5;
    const unsigned long long stride = (unsigned long long)gridDim.x * wpb * per_warp;

    for (unsigned long long j0 = ((unsigned long long)blockIdx.x * wpb + (threadIdx.x >> 5)) * per_warp; j0 < a.B;
         j0 += stride) {
        // every lane of the warp walks (the shuffles need them all); a sub-warp past the batch
        // walks draw j0 again and stores nothing
        const bool active = j0 + sub < a.B;
        const unsigned j = (unsigned)(active ? j0 + sub : j0);
        const double u = draw_uniform(a.seed, j, call, 0);
        double m = __dmul_rn(__dadd_rn(exact_double(j, 0), u), seg);
        unsigned long long leaf;
        float lv = 0.0f;
        if (D == 0) {
            leaf = 0;
            lv = a.t.L[0];
        } else {
            unsigned long long node = 1;
            if (TOP > 0 && top > 0) {
#pragma unroll 1
                for (int lev = 0; lev < top; ++lev) {
                    const double left = s_top[2 * node];
                    if (gt_nonneg(left, m)) {
                        node = 2 * node;
                    } else {
                        m = __dsub_rn(m, left);
                        node = 2 * node + 1;
                    }
                }
            }
            if (!kPre) walk_load<G, S>(a.t, node, first, rounds == 1, lane, w0);
            node = walk_decide<G, S>(node, first, rounds == 1, m, lane, w0, &lv);
            for (int rd = 1; rd < rounds; ++rd) {
                const int k = top > 0 ? kb + (rd < kx) : K;
                const bool lst = rd == rounds - 1;
                // the last round from its leaves alone
                if (TOP > 0 && kLeafRounds && top > 0 && lst && k >= LG && k <= LG + 2) {
                    if (k == LG) node = walk_leaves<G, 0>(a.t, node, m, lane, &lv);
                    else if (k == LG + 1) node = walk_leaves<G, 1>(a.t, node, m, lane, &lv);
                    else node = walk_leaves<G, 2>(a.t, node, m, lane, &lv);
                } else {
                    WalkRegs<S> w;
                    walk_load<G, S>(a.t, node, k, lst, lane, w);
                    node = walk_decide<G, S>(node, k, lst, m, lane, w, &lv);
                }
            }
            leaf = node - n;
        }
        if (leaf >= size) {  // ran past the filled slots: take the last filled slot
            leaf = size - 1;
            lv = a.t.L[leaf];
        }
        if (active) {
            if (lane == 0) {
                a.o.idx[j] = (long long)leaf;
                if (a.o.w) a.o.w[j] = powf(__fdiv_rn(lv, pmin), nbeta);
            }
            gather_row<G, GV>(a.r, a.o, j, leaf, lane, a.vec4);
        }
        // the first round again for the next draw (reloaded here, from L1 or L2, rather than kept
        // in registers through the gather)
        if (kPre && D > 0 && j0 + stride < a.B) walk_load<G, S>(a.t, 1, first, rounds == 1, lane, w0);
    }
}

// The first position p in [lo, hi) with c[p] > m (c non-decreasing, values >= 0), or hi when
// there is none: a 32-way search by the warp -- each round probes 32 evenly spaced entries and
// keeps the bracket that holds the first entry above m (4 rounds for 2^20 entries).
__device__ __forceinline__ unsigned long long first_above(const double *c, unsigned long long lo,
                                                          unsigned long long hi, double m, int lane)
{
    while (true) {
        const unsigned long long len = hi - lo;
        if (len == 0) return hi;
        if (len <= 32) {
            const unsigned long long p = lo + lane;
            const bool pred = p < hi && gt_nonneg(c[p], m);
            const unsigned b = __ballot_sync(kFull, pred);
            return b ? lo + (__ffs(b) - 1) : hi;
        }
        const unsigned long long step = (len + 31) / 32;
        unsigned long long p = lo + (unsigned long long)(lane + 1) * step - 1;
        if (p > hi - 1) p = hi - 1;
        const bool pred = gt_nonneg(c[p], m);
        const unsigned b = __ballot_sync(kFull, pred);
        if (b == 0) return hi;
        const int f = __ffs(b) - 1;
        unsigned long long pf = lo + (unsigned long long)(f + 1) * step - 1;
        if (pf > hi - 1) pf = hi - 1;
        unsigned long long pprev = lo;
        if (f > 0) {
            pprev = lo + (unsigned long long)f * step - 1;
            if (pprev > hi - 1) pprev = hi - 1;
            pprev += 1;
        }
        lo = pprev;
        hi = pf;  // the answer is in [lo, pf]; pf itself is above m
    }
}

// ------------------------------------------------------------------------------------------
// Flat mode ("GPU-Resident Prioritized Experience Replay", Sampling Kernels, Proportional
// steps 3-5): the same draws as proportional mode (counter tag 0, stratified), located by a
// search of the cumulative array C that k_flat_scan built; w = (L[i] / p_min)^-beta; gather.
// ------------------------------------------------------------------------------------------
struct FlatSampleArgs {
    const float *L;
    const double *C;
    const unsigned long long *res;   // [1] T bits, [2] smallest filled leaf bits
    RingRefs r;
    Ctl *ctl;
    unsigned B;
    double inv_b;
    float beta;
    unsigned long long seed;
    SampleOut o;
    int vec4;
};

__global__ void __launch_bounds__(kThreads, 4) k_sample_flat(FlatSampleArgs a)
{
    __shared__ unsigned long long s_call;
    pdl_wait();
    pdl_release();
    if (threadIdx.x == 0) s_call = take_call_number(a.ctl);
    const unsigned long long size = a.ctl->size;
    const double total = __longlong_as_double((long long)a.res[1]);
    const float pmin = __uint_as_float((unsigned)a.res[2]);
    const double seg = a.inv_b != 0.0 ? __dmul_rn(total, a.inv_b) : __ddiv_rn(total, (double)a.B);
    __syncthreads();
    const unsigned long long call = s_call;
    const float nbeta = -a.beta;
    const int lane = threadIdx.x & 31;
    const unsigned wpb = blockDim.x >> 5;
    const unsigned warps_total = gridDim.x * wpb;
    for (unsigned j = blockIdx.x * wpb + (threadIdx.x >> 5); j < a.B; j += warps_total) {
        const double u = draw_uniform(a.seed, j, call, 0);
        const double m = __dmul_rn(__dadd_rn(exact_double(j, 0), u), seg);
        unsigned long long slot = first_above(a.C, 0, size, m, lane);
        if (slot >= size) slot = size - 1;   // ran past the filled slots
        const float lv = a.L[slot];
        if (lane == 0) {
            a.o.idx[j] = (long long)slot;
            if (a.o.w) a.o.w[j] = powf(__fdiv_rn(lv, pmin), nbeta);
        }
        gather_row<32, 4>(a.r, a.o, j, slot, lane, a.vec4);
    }
}

// ------------------------------------------------------------------------------------------
// Rank mode ("Sampling Kernels", Rank-based step 2): rank r is drawn with probability
// r^-alpha / c_size by locating the stratified mass in the CDF c (a 32-way search per warp:
// each round probes 32 evenly spaced entries and keeps the bracket that holds the first
// entry above the mass).  The slot is sorted[r-1]; w = (r / size)^(alpha beta).
// ------------------------------------------------------------------------------------------
struct RankSampleArgs {
    const double *cdf;
    const GuideEntry *guide;         // guide[0 .. guide_k] (see GuideEntry), or null
    unsigned guide_k;
    double guide_delta, guide_inv;
    const unsigned *sorted;          // the slot order, unless order_cur is set:
    const unsigned *vals[2];         //   then vals[*order_cur]
    const unsigned *order_cur;
    RingRefs r;
    Ctl *ctl;
    unsigned B;
    double inv_b;   // 1/B when B is a power of two (exact), else 0
    float ab;  // alpha * beta, the exponent of the closed-form weight
    unsigned long long seed;
    SampleOut o;
    int vec4;
};

__global__ void __launch_bounds__(kThreads, 4) k_sample_rank(RankSampleArgs a)
{
    __shared__ double s_seg;
    __shared__ unsigned long long s_call;
    pdl_wait();
    pdl_release();
    const unsigned *sorted = a.order_cur ? a.vals[*a.order_cur & 1u] : a.sorted;
    const unsigned long long size = a.ctl->size;
    if (threadIdx.x == 0) {
        s_call = take_call_number(a.ctl);
        const double total = __longlong_as_double((long long)a.ctl->rank_total_bits);   // cdf[size]
        s_seg = a.inv_b != 0.0 ? __dmul_rn(total, a.inv_b) : __ddiv_rn(total, (double)a.B);
    }
    __syncthreads();
    const unsigned long long call = s_call;
    const double seg = s_seg;
    const float fsize = (float)size;
    const int lane = threadIdx.x & 31;
    const unsigned wpb = blockDim.x >> 5;
    const unsigned warps_total = gridDim.x * wpb;
    for (unsigned j = blockIdx.x * wpb + (threadIdx.x >> 5); j < a.B; j += warps_total) {
        const double u = draw_uniform(a.seed, j, call, 1);
        const double m = __dmul_rn(__dadd_rn(exact_double(j, 0), u), seg);
        // first position p in [1, size] with cdf[p] > m; size + 1 when there is none.  The
        // guide brackets it: with fl(k delta) <= m < fl((k+1) delta), the rank lies in [r0, r1];
        // when the bucket holds at most three candidates their CDF values come with it, else the
        // search covers that stretch only (the same comparisons either way)
        unsigned long long lo = 1, hi = size + 1, ans = 0;
        bool found = false;
        if (a.guide) {
            // delta is a power of two: m / delta is exact and its truncation is the bucket
            long long k = (long long)__dmul_rn(m, a.guide_inv);
            if (k > (long long)a.guide_k) k = a.guide_k;
            if (k < 0) k = 0;
            const ulonglong2 q0 = __ldg(reinterpret_cast<const ulonglong2 *>(a.guide + k));
            const double2 q1 = __ldg(reinterpret_cast<const double2 *>(a.guide + k) + 1);
            const unsigned long long g0 = (unsigned)q0.x, g1 = (unsigned)(q0.x >> 32);
            if (g1 - g0 <= 3) {
                const double c0 = __longlong_as_double((long long)q0.y);
                const unsigned w = (unsigned)(g1 - g0);
                ans = g0 + (w > 0 && !gt_nonneg(c0, m)) + (w > 1 && !gt_nonneg(q1.x, m)) + (w > 2 && !gt_nonneg(q1.y, m));
                if (ans > hi) ans = hi;
                found = true;
            }
            if (g0 > lo) lo = g0;
            if (g1 < hi) hi = g1;
            if (lo > hi) lo = hi;
        }
        if (!found) ans = first_above(a.cdf, lo, hi, m, lane);
        unsigned long long r = ans > size ? size : ans;
        const unsigned long long slot = sorted[r - 1];
        if (lane == 0) {
            a.o.idx[j] = (long long)slot;
            if (a.o.w) a.o.w[j] = powf(__fdiv_rn((float)r, fsize), a.ab);
        }
        gather_row<32, 4>(a.r, a.o, j, slot, lane, a.vec4);
    }
}

// ------------------------------------------------------------------------------------------
// Uniform mode (the plain replay that prioritized replay replaces): every filled slot weighs 1,
// so the stratified walk is a division.  Draw j: u_j from counter (j, call, tag 2),
// mass_j = (j + u_j) * (size / B), slot floor(mass_j) (clamped to the last filled slot), w = 1.
// One warp per draw, which then gathers the row like the other modes.
// ------------------------------------------------------------------------------------------
struct UniformArgs {
    RingRefs r;
    Ctl *ctl;
    unsigned B;
    double inv_b;   // 1/B when B is a power of two (exact), else 0
    unsigned long long seed;
    SampleOut o;
    int vec4;
};

__global__ void __launch_bounds__(kThreads, 4) k_sample_uniform(UniformArgs a)
{
    __shared__ unsigned long long s_call;
    pdl_wait();
    pdl_release();
    if (threadIdx.x == 0) s_call = take_call_number(a.ctl);
    const unsigned long long size = a.ctl->size;
    const double total = (double)size;
    const double seg = a.inv_b != 0.0 ? __dmul_rn(total, a.inv_b) : __ddiv_rn(total, (double)a.B);
    __syncthreads();
    const unsigned long long call = s_call;
    const int lane = threadIdx.x & 31;
    const unsigned wpb = blockDim.x >> 5;
    const unsigned warps_total = gridDim.x * wpb;
    for (unsigned j = blockIdx.x * wpb + (threadIdx.x >> 5); j < a.B; j += warps_total) {
        const double u = draw_uniform(a.seed, j, call, 2);
        const double m = __dmul_rn(__dadd_rn(exact_double(j, 0), u), seg);
        unsigned long long slot = (unsigned long long)m;   // m >= 0: truncation is the floor
        if (slot >= size) slot = size - 1;
        if (lane == 0) {
            a.o.idx[j] = (long long)slot;
            if (a.o.w) a.o.w[j] = 1.0f;
        }
        gather_row<32, 4>(a.r, a.o, j, slot, lane, a.vec4);
    }
}

// Draws (warps) per CTA of the samplers, measured on GB300 (steps/s of each workload's step):
// 2 for batches of at most 512 or at least 4096 draws (the apex step 35.7K against 34.8K with 8;
// the stress step 20.9K against 20.1K), 8 in between (the dqn step 42.3K against 40.0K with 2
// or 4; the rank step 25.8K against 24.8K).
// CTAs per SM the samplers' grids stop at (larger batches loop over their draws): 16 (24 or 32
// slowed the stress sample from 26.6 to 28.6-32.6 us).
unsigned long long sampler_ctas_per_sm() { return 16; }

int warps_per_cta(unsigned B) { return (B <= 512 || B >= 4096) ? 2 : 8; }

// Batches from which the proportional sampler serves two draws per warp (16 lanes each), and
// four (8 lanes each).
constexpr unsigned kHalfWarpBatch = 4096;
constexpr unsigned kQuarterWarpBatch = 8192;

// Levels of the tree's top that the half- and quarter-warp samplers walk in shared memory (a
// copy of 2^(kTopLevels + 1) nodes a CTA), on trees deeper than kTopMinDepth.
constexpr int kTopLevels = 8, kTopMinDepth = 12;

bool rows_vec4(const RingRefs &r, const SampleOut &o)
{
    if (r.d % 4 != 0 || o.dp % 4 != 0) return false;
    const uintptr_t bits = reinterpret_cast<uintptr_t>(o.states) | reinterpret_cast<uintptr_t>(o.next) |
                           reinterpret_cast<uintptr_t>(r.states) | reinterpret_cast<uintptr_t>(r.next);
    return bits % 16 == 0;
}

}  // namespace

cudaError_t init_sample_kernels(int carveout)
{
    if (carveout < 0) return cudaSuccess;
    cudaError_t e;
    const void *fns[] = {(const void *)k_sample_prop<32, 4, 0>, (const void *)k_sample_prop<16, 4, kTopLevels>,
                         (const void *)k_sample_prop<8, 8, kTopLevels>, (const void *)k_sample_rank,
                         (const void *)k_sample_uniform, (const void *)k_sample_flat};
    for (const void *f : fns) {
        e = cudaFuncSetAttribute(f, cudaFuncAttributePreferredSharedMemoryCarveout, carveout);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t launch_sample_prop(const TreeRefs &t, const RingRefs &r, Ctl *ctl, unsigned B,
                               float beta, unsigned long long seed, const SampleOut &o,
                               int num_sms, cudaStream_t st)
{
    SampleArgs a;
    a.t = t;
    a.r = r;
    a.ctl = ctl;
    a.B = B;
    a.inv_b = (B & (B - 1)) == 0 ? 1.0 / (double)B : 0.0;
    a.beta = beta;
    a.seed = seed;
    a.o = o;
    a.vec4 = rows_vec4(r, o) ? 1 : 0;
    const int wpb = warps_per_cta(B);
    // several draws per warp for large batches, where the walk keeps its number of rounds
    const int r7 = (t.D + 6) / 7, r6 = (t.D + 5) / 6;
    const int per_warp = (B >= kQuarterWarpBatch && r6 == r7) ? 4 : (B >= kHalfWarpBatch && r6 == r7) ? 2 : 1;
    const unsigned long long ctas = (B + wpb * per_warp - 1) / (wpb * per_warp);
    const unsigned grid = (unsigned)std::min<unsigned long long>(ctas, (unsigned long long)num_sms * sampler_ctas_per_sm());
    a.top = per_warp > 1 && t.D > kTopMinDepth ? kTopLevels : 0;
    if (per_warp == 4) return launch_pdl(k_sample_prop<8, 8, kTopLevels>, grid, wpb * 32, 0, st, a);
    if (per_warp == 2) return launch_pdl(k_sample_prop<16, 4, kTopLevels>, grid, wpb * 32, 0, st, a);
    return launch_pdl(k_sample_prop<32, 4, 0>, grid, wpb * 32, 0, st, a);
}

cudaError_t launch_sample_flat(const float *L, const FlatWork &fw, const RingRefs &r, Ctl *ctl, unsigned B,
                               float beta, unsigned long long seed, const SampleOut &o, int num_sms,
                               cudaStream_t st)
{
    FlatSampleArgs a;
    a.L = L;
    a.C = fw.C;
    a.res = fw.res;
    a.r = r;
    a.ctl = ctl;
    a.B = B;
    a.inv_b = (B & (B - 1)) == 0 ? 1.0 / (double)B : 0.0;
    a.beta = beta;
    a.seed = seed;
    a.o = o;
    a.vec4 = rows_vec4(r, o) ? 1 : 0;
    const int wpb = warps_per_cta(B);
    const unsigned long long ctas = (B + wpb - 1) / wpb;
    const unsigned grid = (unsigned)std::min<unsigned long long>(ctas, (unsigned long long)num_sms * sampler_ctas_per_sm());
    return launch_pdl(k_sample_flat, grid, wpb * 32, 0, st, a);
}

cudaError_t launch_sample_uniform(const RingRefs &r, Ctl *ctl, unsigned B, unsigned long long seed,
                                  const SampleOut &o, int num_sms, cudaStream_t st)
{
    UniformArgs a;
    a.r = r;
    a.ctl = ctl;
    a.B = B;
    a.inv_b = (B & (B - 1)) == 0 ? 1.0 / (double)B : 0.0;
    a.seed = seed;
    a.o = o;
    a.vec4 = rows_vec4(r, o) ? 1 : 0;
    const int wpb = warps_per_cta(B);
    const unsigned long long ctas = (B + wpb - 1) / wpb;
    const unsigned grid = (unsigned)std::min<unsigned long long>(ctas, (unsigned long long)num_sms * sampler_ctas_per_sm());
    return launch_pdl(k_sample_uniform, grid, wpb * 32, 0, st, a);
}

cudaError_t launch_sample_rank(const RankWork &w, const unsigned *sorted, const RingRefs &r,
                               Ctl *ctl, unsigned B, float beta, double alpha,
                               unsigned long long seed, const SampleOut &o, int num_sms,
                               cudaStream_t st)
{
    RankSampleArgs a;
    a.cdf = w.cdf;
    a.guide = w.guide;
    a.guide_k = w.guide_k;
    a.guide_delta = w.guide_delta;
    a.guide_inv = w.guide_delta > 0.0 ? 1.0 / w.guide_delta : 0.0;
    a.sorted = sorted;
    a.vals[0] = w.vals[0];
    a.vals[1] = w.vals[1];
    a.order_cur = w.merge_ctl ? w.merge_ctl + 4 : nullptr;
    a.r = r;
    a.ctl = ctl;
    a.B = B;
    a.inv_b = (B & (B - 1)) == 0 ? 1.0 / (double)B : 0.0;
    a.ab = (float)(alpha * (double)beta);
    a.seed = seed;
    a.o = o;
    a.vec4 = rows_vec4(r, o) ? 1 : 0;
    const int wpb = warps_per_cta(B);
    const unsigned long long ctas = (B + wpb - 1) / wpb;
    const unsigned grid = (unsigned)std::min<unsigned long long>(ctas, (unsigned long long)num_sms * sampler_ctas_per_sm());
    return launch_pdl(k_sample_rank, grid, wpb * 32, 0, st, a);
}

}  // namespace gbper
