// k_tree.cu -- insertion and priority-update kernels of the proportional sum/min trees.
//
// "Putting prioritized replay's segment tree on a GPU", Second Port: Make the Update
// GPU-Shaped: write the changed leaves (all independent), then rebuild internal nodes bottom up
// one level at a time, every node of a level being independent.  The race described in "The
// Race Condition Worth Writing Down" (a parent summed before its children are final) is ruled
// out here by construction: a level is finished under a CTA barrier before the level above
// reads it, and nodes shared by several CTAs are only computed by the last CTA to arrive,
// after every other CTA has published its part (fence + arrival ticket, no waiting).
//
// Unlike the post's rebuild, which touches every internal node (O(k + n)), both kernels here
// rebuild only the ancestors of changed leaves: an insertion touches a contiguous leaf range,
// an update a scattered set.  Values are recomputed as S[i] = S[2i] + S[2i+1] (binary64) and
// M[i] = min(M[2i], M[2i+1]) (binary32), so any order of recomputation yields the same bits.
#include "per_internal.cuh"
#include "leaf_pow.cuh"

#include <algorithm>
#include <cstdlib>

namespace gbper {

namespace {

// Tables of the binary32 power (leaf_pow.cuh), uploaded once per device.
__device__ LeafPowTables g_leafpow;

// fl32(pow(raw, alpha)): the double-float evaluation when it decides, else the binary64 pow.
__device__ __forceinline__ float leaf_of(float raw, const LeafPowAlpha &al,
                                         const LeafPowTables &tb = g_leafpow)
{
    float out;
    if (leaf_pow_fast(raw, al, tb, &out)) return out;
    return __double2float_rn(pow((double)raw, al.alpha));
}

constexpr int kThreads = 256;
constexpr int kAddBlockLog = 8;      // leaves per tree CTA in the insertion kernel: 256
constexpr int kTopSpan = 1040;       // widest dirty span the last CTA handles on insertion
constexpr int kMaxTopLog = 10;       // update grid <= 2^10 CTAs

__device__ __forceinline__ float fmin_tree(float a, float b) { return a < b ? a : b; }

__device__ __forceinline__ double ld_sum_cg(const TreeRefs &t, unsigned long long node)
{
    return node >= t.n ? (double)__ldcg(t.L + (node - t.n)) : __ldcg(t.S + node);
}

__device__ __forceinline__ float ld_min_cg(const TreeRefs &t, unsigned long long node)
{
    return node >= t.n ? leaf_min_value(__ldcg(t.L + (node - t.n))) : __ldcg(t.M + node);
}

__device__ __forceinline__ double ld_sum(const TreeRefs &t, unsigned long long node)
{
    return node >= t.n ? (double)t.L[node - t.n] : t.S[node];
}

__device__ __forceinline__ float ld_min(const TreeRefs &t, unsigned long long node)
{
    return node >= t.n ? leaf_min_value(t.L[node - t.n]) : t.M[node];
}

// Arrival ticket: returns true in every thread of the last CTA to arrive.  No CTA waits.  The
// CTA barrier orders every thread's earlier accesses before thread 0's release fence and ticket
// (a fence is cumulative over what happens before it), and the last CTA's thread 0 fences again
// (acquire) before the barrier that lets its other threads read: one fence a CTA instead of one
// a thread (measured on GB300: the dqn step 27.7 against 28.7 us, the apex step 38.9K against
// 38.6K steps/s).
__device__ __forceinline__ bool last_to_arrive(unsigned *ticket)
{
    __shared__ int s_last;
    __syncthreads();
    if (threadIdx.x == 0) {
        asm volatile("fence.acq_rel.gpu;" ::: "memory");
        const unsigned t = atomicAdd(ticket, 1u);
        const int l = t == gridDim.x - 1;
        if (l) asm volatile("fence.acq_rel.gpu;" ::: "memory");
        s_last = l;
    }
    __syncthreads();
    return s_last;
}

__device__ __forceinline__ unsigned block_max_u32(unsigned v)
{
    __shared__ unsigned s_red[kThreads / 32];
    for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
    if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = v;
    __syncthreads();
    if (threadIdx.x < 32) {
        v = threadIdx.x < (blockDim.x >> 5) ? s_red[threadIdx.x] : 0u;
        for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
    }
    __syncthreads();
    return v;  // valid in thread 0
}

// ------------------------------------------------------------------------------------------
// Dirty-range upsweep run by one CTA: the nodes [lo, hi] (offsets within depth L0) are final
// in global memory; recompute every ancestor up to the root.  All loads (the dirty nodes and
// the clean edge siblings of every level) are issued before the first level is combined, so
// the whole climb costs one round trip to L2 plus one barrier per level.
// ------------------------------------------------------------------------------------------
// The same climb for a span of at most 32 nodes, on registers: lane i holds span node i, lane
// l holds the clean edge siblings of depth l, and each level pulls its children by shuffles.
__device__ void top_range_climb_regs(const TreeRefs &t, int L0, unsigned long long lo,
                                     unsigned long long hi, int lane)
{
    const unsigned long long lvl0 = 1ull << L0;
    unsigned long long sp_lo = (lo >> 1) << 1;
    const int w0 = (int)(((hi >> 1) << 1) + 1 - sp_lo + 1);
    double cs = 0.0;
    float cm = 0.0f;
    if (lane < w0) {
        cs = ld_sum_cg(t, lvl0 + sp_lo + lane);
        cm = ld_min_cg(t, lvl0 + sp_lo + lane);
    }
    double exLs = 0.0, exRs = 0.0;
    float exLm = 0.0f, exRm = 0.0f;
    if (lane >= 1 && lane < L0) {  // clean edge siblings of depth `lane`
        const unsigned long long a = lo >> (L0 - lane), b = hi >> (L0 - lane);
        const unsigned long long base = 1ull << lane;
        if (a & 1ull) { exLs = ld_sum_cg(t, base + a - 1); exLm = ld_min_cg(t, base + a - 1); }
        if (!(b & 1ull)) { exRs = ld_sum_cg(t, base + b + 1); exRm = ld_min_cg(t, base + b + 1); }
    }
    // where the range has narrowed to one node, its sibling at depth `lane` is an edge sibling
    double sib1s = 0.0;
    float sib1m = 0.0f;
    if (lane >= 1 && lane < L0) {
        const unsigned long long a_d = lo >> (L0 - lane);
        sib1s = (a_d & 1ull) ? exLs : exRs;
        sib1m = (a_d & 1ull) ? exLm : exRm;
    }
    unsigned long long a = lo, b = hi;
    for (int l = L0; l >= 1; --l) {
        if (a == b) {
            // a single dirty node at depth l: the rest is one path to the root, summed on lane 0
            // from siblings that lane d holds for depth d
            double cur = __shfl_sync(0xffffffffu, cs, (int)(a - sp_lo));
            float curm = __shfl_sync(0xffffffffu, cm, (int)(a - sp_lo));
            unsigned long long node = a;
            for (int d = l; d >= 1; --d) {
                // at depth l the sibling is in the current span; above it, an edge sibling
                const int sl = d == l ? (int)((a ^ 1ull) - sp_lo) : d;
                const double sd = __shfl_sync(0xffffffffu, d == l ? cs : sib1s, sl);
                const float sm = __shfl_sync(0xffffffffu, d == l ? cm : sib1m, sl);
                if (lane == 0) {
                    if (node & 1ull) {
                        cur = sd + cur;
                        curm = fmin_tree(sm, curm);
                    } else {
                        cur = cur + sd;
                        curm = fmin_tree(curm, sm);
                    }
                    node >>= 1;
                    t.S[(1ull << (d - 1)) + node] = cur;
                    t.M[(1ull << (d - 1)) + node] = curm;
                }
            }
            return;
        }
        const unsigned long long pa = a >> 1, pb = b >> 1;   // dirty parents at depth l-1
        const unsigned long long nsp_lo = (pa >> 1) << 1;
        const unsigned long long p = nsp_lo + lane;          // this lane's node at depth l-1
        const int c = (int)(2 * p - sp_lo);
        const int c0 = c >= 0 && c < 32 ? c : 0, c1 = c + 1 >= 0 && c + 1 < 32 ? c + 1 : 0;
        const double l0s = __shfl_sync(0xffffffffu, cs, c0), l1s = __shfl_sync(0xffffffffu, cs, c1);
        const float l0m = __shfl_sync(0xffffffffu, cm, c0), l1m = __shfl_sync(0xffffffffu, cm, c1);
        const int xl = l - 1 >= 1 ? l - 1 : 0;
        const double xLs = __shfl_sync(0xffffffffu, exLs, xl), xRs = __shfl_sync(0xffffffffu, exRs, xl);
        const float xLm = __shfl_sync(0xffffffffu, exLm, xl), xRm = __shfl_sync(0xffffffffu, exRm, xl);
        double ns = 0.0;
        float nm = 0.0f;
        if (p >= pa && p <= pb) {
            ns = l0s + l1s;
            nm = fmin_tree(l0m, l1m);
            t.S[(1ull << (l - 1)) + p] = ns;
            t.M[(1ull << (l - 1)) + p] = nm;
        } else if (l - 1 >= 1 && p == pa - 1 && (pa & 1ull)) {
            ns = xLs;
            nm = xLm;
        } else if (l - 1 >= 1 && p == pb + 1 && !(pb & 1ull)) {
            ns = xRs;
            nm = xRm;
        }
        cs = ns;
        cm = nm;
        sp_lo = nsp_lo;
        a = pa;
        b = pb;
    }
}

__device__ void top_range_upsweep(const TreeRefs &t, int L0, unsigned long long lo,
                                  unsigned long long hi, double *spS0, float *spM0,
                                  double *spS1, float *spM1, double *exS, float *exM)
{
    if (L0 > 0 && L0 <= 32 && ((hi >> 1) << 1) + 2 - ((lo >> 1) << 1) <= 32) {
        if (threadIdx.x < 32) top_range_climb_regs(t, L0, lo, hi, threadIdx.x);
        return;
    }
    // run by warp 0 alone: every level is a handful of nodes, and a warp barrier is far cheaper
    // than a CTA barrier per level
    const int lane = threadIdx.x;
    if (L0 <= 0 || lane >= 32) return;
    const unsigned long long lvl0 = 1ull << L0;
    // span at depth L0: [2(lo>>1), 2(hi>>1)+1]
    unsigned long long sp_lo = (lo >> 1) << 1;
    unsigned long long sp_hi = ((hi >> 1) << 1) + 1;
    const int w0 = (int)(sp_hi - sp_lo + 1);
    for (int i = lane; i < w0; i += 32) {
        spS0[i] = ld_sum_cg(t, lvl0 + sp_lo + i);
        spM0[i] = ld_min_cg(t, lvl0 + sp_lo + i);
    }
    // clean edge siblings of depths L0-1 .. 1: slot 2l (left) and 2l+1 (right)
    for (int l = 1 + lane; l < L0; l += 32) {
        const unsigned long long a = lo >> (L0 - l), b = hi >> (L0 - l);
        const unsigned long long base = 1ull << l;
        if (a & 1ull) { exS[2 * l] = ld_sum_cg(t, base + a - 1); exM[2 * l] = ld_min_cg(t, base + a - 1); }
        if (!(b & 1ull)) { exS[2 * l + 1] = ld_sum_cg(t, base + b + 1); exM[2 * l + 1] = ld_min_cg(t, base + b + 1); }
    }
    __syncwarp();
    double *curS = spS0, *nxtS = spS1;
    float *curM = spM0, *nxtM = spM1;
    unsigned long long a = lo, b = hi;  // dirty range at the current depth
    for (int l = L0; l >= 1; --l) {
        const unsigned long long pa = a >> 1, pb = b >> 1;      // dirty parents at depth l-1
        const int np = (int)(pb - pa + 1);
        // next span at depth l-1 (only needed when l-1 >= 1)
        const unsigned long long nsp_lo = (pa >> 1) << 1;
        const unsigned long long pbase = 1ull << (l - 1);
        for (int i = lane; i < np; i += 32) {
            const unsigned long long p = pa + i;
            const int c = (int)(2 * p - sp_lo);
            const double s = curS[c] + curS[c + 1];
            const float m = fmin_tree(curM[c], curM[c + 1]);
            t.S[pbase + p] = s;
            t.M[pbase + p] = m;
            nxtS[p - nsp_lo] = s;
            nxtM[p - nsp_lo] = m;
        }
        if (lane == 0 && l - 1 >= 1) {
            if (pa & 1ull) { nxtS[0] = exS[2 * (l - 1)]; nxtM[0] = exM[2 * (l - 1)]; }
            if (!(pb & 1ull)) {
                const int r = (int)(pb + 1 - nsp_lo);
                nxtS[r] = exS[2 * (l - 1) + 1];
                nxtM[r] = exM[2 * (l - 1) + 1];
            }
        }
        __syncwarp();
        double *ts = curS; curS = nxtS; nxtS = ts;
        float *tm = curM; curM = nxtM; nxtM = tm;
        sp_lo = nsp_lo;
        a = pa;
        b = pb;
    }
}

// ------------------------------------------------------------------------------------------
// Insertion ("GPU-Resident Prioritized Experience Replay", Experience Insertion).
// CTAs [0, ntree) each own one aligned block of 2^bl leaves that the inserted slot range
// touches: they write the block's new leaves, rebuild its subtree in shared memory and store
// it.  CTAs [ntree, ntree + ncopy) copy the rows.  The last CTA to arrive climbs from the
// dirty block roots to the root and advances the device counters.
// ------------------------------------------------------------------------------------------
struct AddArgs {
    TreeRefs t;
    RingRefs r;
    float *raw_store;
    Ctl *ctl;
    DirtyRefs dirty;   // rank mode: slots written are marked for the next order merge
    unsigned long long count, k0;
    const float *states, *next;
    const unsigned *actions;
    const float *rewards;
    const unsigned char *dones;
    const float *prio;
    double alpha, eps;
    LeafPowAlpha lp;
    int proportional;
    int bl;            // log2 leaves per tree block
    unsigned ntree;    // tree CTAs (upper bound over cursor positions)
    unsigned ncopy;    // row-copy CTAs
    int vec4;          // rows copy as float4
    const double *rank_cdf;   // rank mode: the rank CDF, whose value at the new size the last CTA keeps
};

struct AddGeom {
    unsigned long long s0, endA, lenB;  // range A = [s0, endA), range B = [0, lenB)
    unsigned long long blkA0, nA, nB;
};

__device__ __forceinline__ AddGeom add_geometry(const AddArgs &a, unsigned long long cursor)
{
    AddGeom g;
    const unsigned long long C = a.r.capacity;
    const unsigned long long cnt = a.count - a.k0;
    g.s0 = (cursor + a.k0) % C;
    g.endA = min(g.s0 + cnt, C);
    g.lenB = cnt - (g.endA - g.s0);
    g.blkA0 = g.s0 >> a.bl;
    g.nA = ((g.endA - 1) >> a.bl) - g.blkA0 + 1;
    g.nB = g.lenB ? ((g.lenB - 1) >> a.bl) + 1 : 0;
    return g;
}

__device__ __forceinline__ void copy_row(const AddArgs &a, unsigned long long k,
                                         unsigned long long slot, int lane0, int nlanes)
{
    const unsigned d = a.r.d;
    if (a.vec4) {
        const unsigned d4 = d >> 2;
        const float4 *s = reinterpret_cast<const float4 *>(a.states + k * d);
        const float4 *x = reinterpret_cast<const float4 *>(a.next + k * d);
        float4 *ds = reinterpret_cast<float4 *>(a.r.states + slot * d);
        float4 *dx = reinterpret_cast<float4 *>(a.r.next + slot * d);
        for (unsigned c = lane0; c < d4; c += nlanes) {
            ds[c] = __ldg(s + c);
            dx[c] = __ldg(x + c);
        }
    } else {
        for (unsigned c = lane0; c < d; c += nlanes) {
            a.r.states[slot * d + c] = __ldg(a.states + k * d + c);
            a.r.next[slot * d + c] = __ldg(a.next + k * d + c);
        }
    }
}

// The inserted rows land on at most two contiguous slot ranges, [s0, endA) and [0, lenB), so
// each array is copied as one or two flat streams: thread t moves elements t, t + stride, ...,
// four of them in flight per pass (float4 for the state rows when their layout allows).
template <typename V>
__device__ __forceinline__ void copy_flat(V *dst, const V *src, unsigned long long lenA,
                                          unsigned long long total, unsigned long long dstA,
                                          unsigned long long t0, unsigned long long stride)
{
    for (unsigned long long e0 = t0; e0 < total; e0 += 4 * stride) {
        V v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const unsigned long long e = e0 + u * stride;
            if (e < total) v[u] = __ldg(src + e);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const unsigned long long e = e0 + u * stride;
            if (e < total) dst[e < lenA ? dstA + e : e - lenA] = v[u];
        }
    }
}

// One pass over the inserted rows: a thread issues the loads of its whole share (states and
// next_states elements and the scalar fields, kCopyU of each) before its first store, so the
// copy costs one memory round trip per kCopyU x stride elements.  Range A of the ring starts at
// slot s0 and holds lenA rows; the rest wraps to slot 0.
constexpr int kCopyU = 4;

template <typename V>
__device__ __forceinline__ void copy_rows_pass(const AddArgs &a, const V *srcS, const V *srcN, V *dstS,
                                               V *dstN, unsigned per_row, unsigned long long s0,
                                               unsigned long long lenA, unsigned long long cnt,
                                               unsigned long long t0, unsigned long long stride)
{
    const unsigned long long nv = cnt * per_row;   // elements of states (and of next_states)
    const unsigned long long lenAv = lenA * per_row, s0v = s0 * per_row;
    const unsigned long long total = nv > cnt ? nv : cnt;
    const unsigned *srcA = a.actions + a.k0;
    const float *srcR = a.rewards + a.k0;
    const unsigned char *srcD = a.dones + a.k0;
    for (unsigned long long e0 = t0; e0 < total; e0 += kCopyU * stride) {
        V vs[kCopyU], vn[kCopyU];
        unsigned va[kCopyU];
        float vr[kCopyU];
        unsigned char vd[kCopyU];
#pragma unroll
        for (int u = 0; u < kCopyU; ++u) {
            const unsigned long long e = e0 + u * stride;
            if (e < nv) {
                vs[u] = __ldg(srcS + e);
                vn[u] = __ldg(srcN + e);
            }
            if (e < cnt) {
                va[u] = __ldg(srcA + e);
                vr[u] = __ldg(srcR + e);
                vd[u] = __ldg(srcD + e);
            }
        }
#pragma unroll
        for (int u = 0; u < kCopyU; ++u) {
            const unsigned long long e = e0 + u * stride;
            if (e < nv) {
                const unsigned long long o = e < lenAv ? s0v + e : e - lenAv;
                dstS[o] = vs[u];
                dstN[o] = vn[u];
            }
            if (e < cnt) {
                const unsigned long long o = e < lenA ? s0 + e : e - lenA;
                a.r.actions[o] = va[u];
                a.r.rewards[o] = vr[u];
                a.r.dones[o] = vd[u];
            }
        }
    }
}

__device__ __forceinline__ void copy_rows_flat(const AddArgs &a, const AddGeom &g,
                                               unsigned long long t0, unsigned long long stride)
{
    const unsigned long long cnt = a.count - a.k0;
    const unsigned long long lenA = g.endA - g.s0;
    const unsigned d = a.r.d;
    if (d && a.vec4) {
        const unsigned d4 = d >> 2;
        copy_rows_pass(a, reinterpret_cast<const float4 *>(a.states) + a.k0 * d4,
                       reinterpret_cast<const float4 *>(a.next) + a.k0 * d4, reinterpret_cast<float4 *>(a.r.states),
                       reinterpret_cast<float4 *>(a.r.next), d4, g.s0, lenA, cnt, t0, stride);
    } else {
        copy_rows_pass(a, d ? a.states + a.k0 * d : nullptr, d ? a.next + a.k0 * d : nullptr, a.r.states, a.r.next,
                       d, g.s0, lenA, cnt, t0, stride);
    }
}

__global__ void __launch_bounds__(kThreads) k_add(AddArgs a)
{
    __shared__ LeafPowTables s_lp;
    if (blockIdx.x < a.ntree && a.prio && a.proportional) {
        // the power's tables (constant since the library loaded), staged before the wait
        const unsigned *src = reinterpret_cast<const unsigned *>(&g_leafpow);
        unsigned *dst = reinterpret_cast<unsigned *>(&s_lp);
        for (int i = threadIdx.x; i < (int)(sizeof(LeafPowTables) / 4); i += blockDim.x) dst[i] = src[i];
        __syncthreads();
    }
    pdl_wait();
    pdl_release();
    const unsigned long long cursor = a.ctl->cursor;
    const float max_prev = __uint_as_float(a.ctl->max_raw_bits);
    const float max_leaf = __uint_as_float(a.ctl->max_leaf_bits);
    const unsigned long long size0 = a.ctl->size;
    const unsigned long long C = a.r.capacity;
    const AddGeom g = add_geometry(a, cursor);
    const int tid = threadIdx.x;
    // Every CTA arrives once; the last to arrive climbs and advances the counters, which every
    // CTA has read above before it arrives.  Copy CTAs arrive before copying, so the climb does
    // not wait for the rows (the next kernel waits for this whole grid), unless rows overwritten
    // within this call (k < k0) feed the running maximum through them.
    const bool copies_late = a.k0 > 0 && a.prio;
    bool last = false;

    if (blockIdx.x < a.ntree) {
        const unsigned b = blockIdx.x;
        long long blk = -1;
        if (b < g.nA) blk = (long long)(g.blkA0 + b);
        else if (b < g.nA + g.nB) blk = (long long)(b - g.nA);
        unsigned mymax = 0;
        if (blk >= 0) {
            const int bsz = 1 << a.bl;
            float leaf = 0.0f;
            const unsigned long long s = ((unsigned long long)blk << a.bl) + tid;
            if (tid < bsz) {
                const bool inA = s >= g.s0 && s < g.endA;
                const bool inB = s < g.lenB;
                if (inA || inB) {
                    const unsigned long long off = inA ? s - g.s0 : s + (C - g.s0);
                    const unsigned long long k = a.k0 + off;
                    const float raw = a.prio ? prio_to_raw(__ldg(a.prio + k), a.eps, max_prev) : max_prev;
                    mymax = __float_as_uint(raw);
                    if (a.proportional) {
                        leaf = a.prio ? leaf_of(raw, a.lp, s_lp) : max_leaf;
                        a.t.L[s] = leaf;
                    } else if (a.raw_store) {   // rank mode (uniform mode keeps no priorities)
                        const float old = a.raw_store[s];
                        a.raw_store[s] = raw;
                        mark_dirty(a.dirty, s, old);
                    }
                } else if (a.proportional) {
                    leaf = a.t.L[s];
                }
            }
            if (a.proportional && a.t.S) {   // flat mode keeps leaves only
                // the block's subtree: five levels inside each warp by shuffles, the rest on
                // warp 0 from the warps' sums
                const unsigned long long first = a.t.n + ((unsigned long long)blk << a.bl);
                const int lane = tid & 31, warp = tid >> 5;
                double sv = tid < bsz ? (double)leaf : 0.0;
                float mv = tid < bsz ? leaf_min_value(leaf) : __int_as_float(0x7f800000);
                const int hw = a.bl < 5 ? a.bl : 5;
                for (int h = 1; h <= hw; ++h) {
                    const double os = __shfl_down_sync(0xffffffffu, sv, 1 << (h - 1));
                    const float om = __shfl_down_sync(0xffffffffu, mv, 1 << (h - 1));
                    sv = sv + os;
                    mv = fmin_tree(mv, om);
                    if ((tid & ((1 << h) - 1)) == 0 && tid < bsz) {
                        const unsigned long long node = (first >> h) + (tid >> h);
                        a.t.S[node] = sv;
                        a.t.M[node] = mv;
                    }
                }
                if (a.bl > 5) {
                    __shared__ double s_ws[kThreads / 32];
                    __shared__ float s_wm[kThreads / 32];
                    if (lane == 0) {
                        s_ws[warp] = sv;
                        s_wm[warp] = mv;
                    }
                    __syncthreads();
                    if (warp == 0) {
                        const int nw = bsz >> 5;
                        sv = lane < nw ? s_ws[lane] : 0.0;
                        mv = lane < nw ? s_wm[lane] : __int_as_float(0x7f800000);
                        for (int h = 6; h <= a.bl; ++h) {
                            const double os = __shfl_down_sync(0xffffffffu, sv, 1 << (h - 6));
                            const float om = __shfl_down_sync(0xffffffffu, mv, 1 << (h - 6));
                            sv = sv + os;
                            mv = fmin_tree(mv, om);
                            if ((lane & ((1 << (h - 5)) - 1)) == 0 && lane < nw) {
                                const unsigned long long node = (first >> h) + (lane >> (h - 5));
                                a.t.S[node] = sv;
                                a.t.M[node] = mv;
                            }
                        }
                    }
                }
            }
        }
        const unsigned bm = block_max_u32(mymax);
        if (tid == 0 && bm) atomicMax(&a.ctl->add_max_bits, bm);
        last = last_to_arrive(&a.ctl->ticket_add);
    } else {
        if (!copies_late) last = last_to_arrive(&a.ctl->ticket_add);
        // rows that a later row of the same call overwrites still count toward the running
        // maximum, as if they had been inserted one after another
        if (copies_late) {
            unsigned mymax = 0;
            const unsigned long long t0 = (unsigned long long)(blockIdx.x - a.ntree) * kThreads + tid;
            for (unsigned long long k = t0; k < a.k0; k += (unsigned long long)a.ncopy * kThreads)
                mymax = max(mymax, __float_as_uint(prio_to_raw(__ldg(a.prio + k), a.eps, max_prev)));
            const unsigned bm = block_max_u32(mymax);
            if (tid == 0 && bm) atomicMax(&a.ctl->add_max_bits, bm);
        }
        copy_rows_flat(a, g, (unsigned long long)(blockIdx.x - a.ntree) * kThreads + tid,
                       (unsigned long long)a.ncopy * kThreads);
        if (copies_late) last = last_to_arrive(&a.ctl->ticket_add);
    }

    if (last) {
        unsigned call_max = 0;
        if (tid == 0) call_max = __ldcg(&a.ctl->add_max_bits);   // in flight during the climb
        if (a.proportional && a.t.S) {
            __shared__ double s_spS0[kTopSpan], s_spS1[kTopSpan];
            __shared__ float s_spM0[kTopSpan], s_spM1[kTopSpan];
            __shared__ double s_exS[64];
            __shared__ float s_exM[64];
            const int L0 = a.t.D - a.bl;
            top_range_upsweep(a.t, L0, g.blkA0, g.blkA0 + g.nA - 1, s_spS0, s_spM0, s_spS1,
                              s_spM1, s_exS, s_exM);
            if (g.nB) {
                __syncwarp();
                top_range_upsweep(a.t, L0, 0, g.nB - 1, s_spS0, s_spM0, s_spS1, s_spM1, s_exS,
                                  s_exM);
            }
        }
        if (tid == 0) {
            Ctl *c = a.ctl;
            fold_running_max(c, call_max, a.alpha);
            c->add_max_bits = 0;
            c->cursor = (cursor + a.count) % C;
            const unsigned long long sz = size0 + a.count < C ? size0 + a.count : C;
            c->size = sz;
            if (a.rank_cdf && sz != size0) c->rank_total_bits = (unsigned long long)__double_as_longlong(a.rank_cdf[sz]);
            c->ticket_add = 0;
        }
    }
}

// ---- bulk insertion: rows + leaves, then a full level-by-level rebuild -------------------

__global__ void __launch_bounds__(kThreads) k_add_bulk_rows(AddArgs a)
{
    pdl_wait();
    pdl_release();
    const unsigned long long cursor = a.ctl->cursor;
    const float max_prev = __uint_as_float(a.ctl->max_raw_bits);
    const unsigned long long C = a.r.capacity;
    const unsigned long long cnt = a.count - a.k0;
    const unsigned long long s0 = (cursor + a.k0) % C;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const unsigned long long wglob = (unsigned long long)blockIdx.x * (kThreads / 32) + warp;
    const unsigned long long wtotal = (unsigned long long)gridDim.x * (kThreads / 32);
    unsigned mymax = 0;
    if (a.prio) {  // overwritten rows of this call still count toward the running maximum
        const unsigned long long t0 = (unsigned long long)blockIdx.x * kThreads + threadIdx.x;
        for (unsigned long long k = t0; k < a.k0; k += (unsigned long long)gridDim.x * kThreads)
            mymax = max(mymax, __float_as_uint(prio_to_raw(__ldg(a.prio + k), a.eps, max_prev)));
    }
    for (unsigned long long o = wglob; o < cnt; o += wtotal) {
        const unsigned long long k = a.k0 + o;
        const unsigned long long slot = (s0 + o) % C;
        if (a.r.d) copy_row(a, k, slot, lane, 32);
        if (lane == 0) {
            a.r.actions[slot] = __ldg(a.actions + k);
            a.r.rewards[slot] = __ldg(a.rewards + k);
            a.r.dones[slot] = __ldg(a.dones + k);
            const float raw = a.prio ? prio_to_raw(__ldg(a.prio + k), a.eps, max_prev) : max_prev;
            mymax = max(mymax, __float_as_uint(raw));
            if (a.proportional)
                a.t.L[slot] = a.prio ? leaf_of(raw, a.lp) : __uint_as_float(a.ctl->max_leaf_bits);
            else if (a.raw_store) a.raw_store[slot] = raw;
        }
    }
    const unsigned bm = block_max_u32(mymax);
    if (threadIdx.x == 0 && bm) atomicMax(&a.ctl->add_max_bits, bm);
}

// ---- full rebuild of both trees ("Putting prioritized replay's segment tree on a GPU", Second
// Port: every node from its two children, level after level) ---------------------------------
// One CTA of 256 threads builds the 11 levels above 2048 consecutive nodes of depth cd (the
// leaves when cd = D): each thread combines its 8 inputs on registers for 3 levels (stored as
// 32-, 16- and 8-byte vectors), the next 5 levels run on warp shuffles and the last 3 on warp 0.
// When the CTA roots number at most 2048, the last CTA to arrive builds the levels above them the
// same way (or in shared memory when they are fewer than 256) up to the root; otherwise the host
// launches the next 11 levels.  A tree with fewer than 2048 leaves is built by one CTA.
// In the large-batch update the leaf level also applies the batch: a slot whose winner word is
// set takes the winning entry's priority (and the word is cleared) before it enters the sums.
constexpr int kRbIn = 2048;   // inputs per CTA
constexpr int kRbLog = 11;

struct RebuildArgs {
    TreeRefs t;
    Ctl *ctl;
    int cd;            // depth of this launch's inputs
    unsigned *win;     // large-batch update: winner words (entry + 1, or 0); null otherwise
    const float *td;
    double eps;
    LeafPowAlpha lp;
    int fold;          // fold batch_max_bits into the running maximum once the root is built
    double alpha;
    CrowdRefs crowd;   // hist non-null: the fold also reports (and clears) the subtree counts
};

// binary32 -> binary64 on the integer pipe for leaves (0, +inf or normal numbers: a leaf is at
// least eps^alpha, which per_create keeps >= the smallest normal binary32)
__device__ __forceinline__ double leaf_to_double(float f)
{
    const unsigned b = __float_as_uint(f);
    const unsigned e = b >> 23;
    if (b == 0u) return 0.0;
    if (e == 0u) return (double)f;   // subnormal: not a leaf value, kept exact anyway
    const unsigned long long e64 = e == 255u ? 2047ull : (unsigned long long)(e + (1023 - 127));
    return __longlong_as_double((long long)((e64 << 52) | ((unsigned long long)(b & 0x7fffffu) << 29)));
}

// The leaf value of slot i under the large-batch update: the winning entry's leaf when the
// slot's winner word w is set (then written back, word cleared), else the stored leaf.  `tdv`
// is the winning entry's TD error, loaded by the caller (all of a thread's loads go out first).
__device__ __forceinline__ float applied_leaf(const RebuildArgs &a, unsigned long long i, float stored,
                                              unsigned w, float tdv, float max_prev)
{
    if (w == 0u) return stored;
    const float leaf = leaf_of(td_to_raw(tdv, a.eps, max_prev), a.lp);
    a.t.L[i] = leaf;
    a.win[i] = 0u;
    return leaf;
}

// Sums of 8 leaves for the three register levels as exact integers: each leaf (0 or a normal
// binary32) is its 24-bit significand shifted by (exponent - elo), elo the smallest exponent among
// them; when the exponents span at most 26 binades every partial sum is below 2^53, so it is the
// exact value a binary64 add of the two children gives.  Returns false (sums unset) otherwise, or
// for an infinite or subnormal leaf.
__device__ __forceinline__ bool exact_leaf_sums(const float *lf, unsigned long long *isum, int &elo)
{
    int lo = 255, hi = 0;
    bool special = false;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const unsigned b = __float_as_uint(lf[k]);
        const int e = (int)(b >> 23);
        if (b != 0u) {
            lo = min(lo, e);
            hi = max(hi, e);
            special |= e == 0 || e == 255;
        }
    }
    if (special || (hi >= lo && hi - lo > 26)) return false;
    if (hi < lo) lo = 127;   // every leaf is 0
    unsigned long long iv[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const unsigned b = __float_as_uint(lf[k]);
        iv[k] = b ? (unsigned long long)((b & 0x7fffffu) | 0x800000u) << ((int)(b >> 23) - lo) : 0ull;
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) isum[k] = iv[2 * k] + iv[2 * k + 1];
    isum[4] = isum[0] + isum[1];
    isum[5] = isum[2] + isum[3];
    isum[6] = isum[4] + isum[5];
    elo = lo;
    return true;
}

// x * 2^(elo - 150) for an integer x < 2^53: exact, assembled on the integer pipe
__device__ __forceinline__ double fixed_to_double_exact(unsigned long long x, int elo)
{
    if (x == 0ull) return 0.0;
    const int p = 63 - __clzll((long long)x);
    const unsigned long long mant = x << (52 - p);
    const unsigned long long e = (unsigned long long)(p + elo - 150 + 1023);
    return __longlong_as_double((long long)((e << 52) | (mant & ((1ull << 52) - 1ull))));
}

template <int CNT>
__device__ __forceinline__ void store_run(const TreeRefs &t, unsigned long long node, const double *v,
                                          const float *m)
{
    if constexpr (CNT == 4) {
        reinterpret_cast<double2 *>(t.S + node)[0] = make_double2(v[0], v[1]);
        reinterpret_cast<double2 *>(t.S + node)[1] = make_double2(v[2], v[3]);
        *reinterpret_cast<float4 *>(t.M + node) = make_float4(m[0], m[1], m[2], m[3]);
    } else if constexpr (CNT == 2) {
        *reinterpret_cast<double2 *>(t.S + node) = make_double2(v[0], v[1]);
        *reinterpret_cast<float2 *>(t.M + node) = make_float2(m[0], m[1]);
    } else {
        t.S[node] = v[0];
        t.M[node] = m[0];
    }
}

// Builds the log2(256 PER) levels above the 256 PER nodes of depth cd that start at `base`
// (PER per thread, consecutive); the top node ends in thread 0's registers and in S/M.  Inputs
// are leaves (with the update applied when a.win is set) or S/M nodes (read from L2 when `cg`,
// i.e. written by other CTAs of this launch).
template <int PER>
__device__ __forceinline__ void build_block(const RebuildArgs &a, unsigned long long base, bool leaves,
                                            bool cg, float max_prev, unsigned char *smem)
{
    const TreeRefs &t = a.t;
    const int tid = threadIdx.x;
    const unsigned long long i0 = base + (unsigned long long)PER * tid;
    double v[PER];
    float m[PER];
    bool exact = false;             // leaves whose three register levels are exact integer sums
    unsigned long long isum[7] = {}; // those sums: level 1 [0..3], level 2 [4..5], level 3 [6]
    int elo = 0;                    // their unit is 2^(elo - 150)
    if (leaves) {
        float lf[PER];
        const unsigned long long l0 = i0 - t.n;
        if constexpr (PER == 8) {
            const float4 x = reinterpret_cast<const float4 *>(t.L + l0)[0];
            const float4 y = reinterpret_cast<const float4 *>(t.L + l0)[1];
            lf[0] = x.x; lf[1] = x.y; lf[2] = x.z; lf[3] = x.w;
            lf[4] = y.x; lf[5] = y.y; lf[6] = y.z; lf[7] = y.w;
            if (a.win) {
                // the warp's winners (slots whose word is set) go into a list in shared memory
                // and are computed 32 at a time, so the leaf power runs on full warps
                const uint4 wx = reinterpret_cast<const uint4 *>(a.win + l0)[0];
                const uint4 wy = reinterpret_cast<const uint4 *>(a.win + l0)[1];
                const unsigned w[8] = {wx.x, wx.y, wx.z, wx.w, wy.x, wy.y, wy.z, wy.w};
                const int lane = tid & 31, wb = (tid >> 5) * 256;
                unsigned char *s_pos = smem;                                          // [2048]
                unsigned *s_w = reinterpret_cast<unsigned *>(smem + 2048);            // [2048]
                float *s_lv = reinterpret_cast<float *>(smem + 2048 + 4 * 2048);      // [2048]
                int cnt = 0;
#pragma unroll
                for (int k = 0; k < 8; ++k) cnt += w[k] != 0u;
                int incl = cnt;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int y = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl += y;
                }
                const int total = __shfl_sync(0xffffffffu, incl, 31);
                if (total > 0) {
                    int off = wb + incl - cnt;
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        if (w[k]) {
                            s_pos[off] = (unsigned char)(lane * 8 + k);
                            s_w[off] = w[k];
                            ++off;
                        }
                    }
                    __syncwarp();
                    const unsigned long long wl0 = l0 - 8ull * lane;   // the warp's first slot
                    for (int r = lane; r < total; r += 32) {
                        const int pos = s_pos[wb + r];
                        const unsigned ww = s_w[wb + r];
                        s_lv[wb + pos] = applied_leaf(a, wl0 + pos, 0.0f, ww, __ldg(a.td + (ww - 1u)), max_prev);
                    }
                    __syncwarp();
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        if (w[k]) lf[k] = s_lv[wb + lane * 8 + k];
                }
            }
        } else {
#pragma unroll
            for (int k = 0; k < PER; ++k) {
                lf[k] = t.L[l0 + k];
                if (a.win) {
                    const unsigned w = a.win[l0 + k];
                    lf[k] = applied_leaf(a, l0 + k, lf[k], w, w ? __ldg(a.td + (w - 1u)) : 0.0f, max_prev);
                }
            }
        }
#pragma unroll
        for (int k = 0; k < PER; ++k) {
            v[k] = leaf_to_double(lf[k]);
            m[k] = leaf_min_value(lf[k]);
        }
        if constexpr (PER == 8) exact = exact_leaf_sums(lf, isum, elo);
    } else {
#pragma unroll
        for (int k = 0; k < PER; k += 2 > PER ? 1 : 2) {
            if constexpr (PER == 1) {
                v[0] = cg ? __ldcg(t.S + i0) : t.S[i0];
            } else {
                const double2 d = cg ? __ldcg(reinterpret_cast<const double2 *>(t.S + i0 + k))
                                     : *reinterpret_cast<const double2 *>(t.S + i0 + k);
                v[k] = d.x;
                v[k + 1] = d.y;
            }
        }
#pragma unroll
        for (int k = 0; k < PER; ++k) m[k] = cg ? __ldcg(t.M + i0 + k) : t.M[i0 + k];
    }
    // levels on registers: after step r the thread holds PER >> r nodes at (i0 >> r); for 8 leaves
    // whose exponents span at most 26 binades the sums are exact integers (converted on the
    // integer pipe), else binary64 adds
    int lv = 0;
    bool done = false;
    if constexpr (PER == 8) {
        if (exact) {
            double d[7];
#pragma unroll
            for (int k = 0; k < 7; ++k) d[k] = fixed_to_double_exact(isum[k], elo);
#pragma unroll
            for (int k = 0; k < 4; ++k) m[k] = fmin_tree(m[2 * k], m[2 * k + 1]);
            store_run<4>(t, i0 >> 1, d, m);
            m[0] = fmin_tree(m[0], m[1]);
            m[1] = fmin_tree(m[2], m[3]);
            store_run<2>(t, i0 >> 2, d + 4, m);
            m[0] = fmin_tree(m[0], m[1]);
            store_run<1>(t, i0 >> 3, d + 6, m);
            v[0] = d[6];
            lv = 3;
            done = true;
        }
    }
    if (!done) {
#pragma unroll
        for (int cnt = PER / 2; cnt >= 1; cnt /= 2) {
            ++lv;
#pragma unroll
            for (int k = 0; k < cnt; ++k) {
                v[k] = v[2 * k] + v[2 * k + 1];
                m[k] = fmin_tree(m[2 * k], m[2 * k + 1]);
            }
            const unsigned long long node = i0 >> lv;
            if (cnt == 4) store_run<4>(t, node, v, m);
            else if (cnt == 2) store_run<2>(t, node, v, m);
            else store_run<1>(t, node, v, m);
        }
    }
    double sv = v[0];
    float mv = m[0];
    const unsigned long long pr = i0 >> lv;   // = (base >> lv) + tid
    const int lane = tid & 31, warp = tid >> 5;
#pragma unroll
    for (int h = 1; h <= 5; ++h) {
        const double os = __shfl_down_sync(0xffffffffu, sv, 1 << (h - 1));
        const float om = __shfl_down_sync(0xffffffffu, mv, 1 << (h - 1));
        sv = sv + os;
        mv = fmin_tree(mv, om);
        if ((lane & ((1 << h) - 1)) == 0) {
            t.S[pr >> h] = sv;
            t.M[pr >> h] = mv;
        }
    }
    __shared__ double s_wv[kThreads / 32];
    __shared__ float s_wm[kThreads / 32];
    if (lane == 0) {
        s_wv[warp] = sv;
        s_wm[warp] = mv;
    }
    __syncthreads();
    if (warp == 0) {
        constexpr int nw = kThreads / 32;
        sv = lane < nw ? s_wv[lane] : 0.0;
        mv = lane < nw ? s_wm[lane] : __int_as_float(0x7f800000);
        const unsigned long long pw = (pr >> 5) - (tid >> 5) + lane;   // the warp roots' depth
#pragma unroll
        for (int h = 1; h <= 3; ++h) {
            const double os = __shfl_down_sync(0xffffffffu, sv, 1 << (h - 1));
            const float om = __shfl_down_sync(0xffffffffu, mv, 1 << (h - 1));
            sv = sv + os;
            mv = fmin_tree(mv, om);
            if ((lane & ((1 << h) - 1)) == 0 && lane < nw) {
                t.S[pw >> h] = sv;
                t.M[pw >> h] = mv;
            }
        }
    }
}

// Every level above the w nodes (a power of two below 256 when called for the top, below 2048
// for a small tree) of one depth starting at node `first`, in shared memory.
__device__ void rebuild_smem(const RebuildArgs &a, unsigned long long first, int w, bool cg, float max_prev,
                             unsigned char *smem)
{
    const TreeRefs &t = a.t;
    double *s_v = reinterpret_cast<double *>(smem);                  // [kRbIn]
    float *s_m = reinterpret_cast<float *>(smem + 8 * kRbIn);        // [kRbIn]
    constexpr int kPer = kRbIn / 2 / kThreads;
    for (int i = threadIdx.x; i < w; i += kThreads) {
        const unsigned long long node = first + i;
        if (node >= t.n) {
            float lf = t.L[node - t.n];
            if (a.win) {
                const unsigned w = a.win[node - t.n];
                lf = applied_leaf(a, node - t.n, lf, w, w ? __ldg(a.td + (w - 1u)) : 0.0f, max_prev);
            }
            s_v[i] = leaf_to_double(lf);
            s_m[i] = leaf_min_value(lf);
        } else {
            s_v[i] = cg ? __ldcg(t.S + node) : t.S[node];
            s_m[i] = cg ? __ldcg(t.M + node) : t.M[node];
        }
    }
    for (int h = 1; (1 << h) <= w; ++h) {
        const int cnt = w >> h;
        double v[kPer];
        float m[kPer];
        __syncthreads();
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
            const int i = threadIdx.x + k * kThreads;
            if (i < cnt) {
                v[k] = s_v[2 * i] + s_v[2 * i + 1];
                m[k] = fmin_tree(s_m[2 * i], s_m[2 * i + 1]);
            }
        }
        __syncthreads();
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
            const int i = threadIdx.x + k * kThreads;
            if (i < cnt) {
                s_v[i] = v[k];
                s_m[i] = m[k];
                const unsigned long long node = (first >> h) + i;
                t.S[node] = v[k];
                t.M[node] = m[k];
            }
        }
    }
}

// The last CTA, once the root is built (every thread of it calls this).
__device__ __forceinline__ void rebuild_fold(const RebuildArgs &a)
{
    if (a.fold && threadIdx.x == 0) {
        fold_running_max(a.ctl, __ldcg(&a.ctl->batch_max_bits), a.alpha);
        a.ctl->batch_max_bits = 0;
    }
    if (a.crowd.hist) {   // the most entries in one subtree, to the host; the counts cleared
        __shared__ unsigned s_cmax;
        if (threadIdx.x == 0) s_cmax = 0;
        __syncthreads();
        unsigned m = 0;
        for (unsigned i = threadIdx.x; i < a.crowd.nsub; i += blockDim.x) {
            m = max(m, __ldcg(a.crowd.hist + i));
            a.crowd.hist[i] = 0u;
        }
        for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
        if ((threadIdx.x & 31) == 0 && m) atomicMax(&s_cmax, m);
        __syncthreads();
        if (threadIdx.x == 0 && a.crowd.host)
            *(volatile unsigned *)a.crowd.host = crowd_report(a.ctl, 31 - __clz(a.crowd.nsub), s_cmax);
    }
}

__global__ void __launch_bounds__(kThreads) k_rebuild_tree(RebuildArgs a)
{
    pdl_wait();
    pdl_release();
    const int cd = a.cd;
    // winner lists of the leaf level, or the top levels' nodes (24 KiB)
    __shared__ __align__(16) unsigned char s_buf[12 * kRbIn];
    const float max_prev = __uint_as_float(a.ctl->max_raw_bits);   // folded only at the end
    if ((1ull << cd) < (unsigned long long)kRbIn) {                  // small tree: one CTA
        rebuild_smem(a, 1ull << cd, 1 << cd, false, max_prev, s_buf);
        rebuild_fold(a);
        return;
    }
    const unsigned long long base = (1ull << cd) + (unsigned long long)blockIdx.x * kRbIn;
    build_block<8>(a, base, cd == a.t.D, false, max_prev, s_buf);
    const unsigned roots = gridDim.x;
    if (roots == 1) {
        rebuild_fold(a);
        return;
    }
    if (roots <= (unsigned)kRbIn && last_to_arrive(&a.ctl->ticket_rebuild)) {
        if (threadIdx.x == 0) a.ctl->ticket_rebuild = 0;
        const unsigned long long first = 1ull << (cd - kRbLog);
        __syncthreads();   // the block builder's shared words are reused below
        if (roots == 2048) build_block<8>(a, first, false, true, max_prev, s_buf);
        else if (roots == 1024) build_block<4>(a, first, false, true, max_prev, s_buf);
        else if (roots == 512) build_block<2>(a, first, false, true, max_prev, s_buf);
        else if (roots == 256) build_block<1>(a, first, false, true, max_prev, s_buf);
        else rebuild_smem(a, first, (int)roots, true, max_prev, s_buf);
        rebuild_fold(a);
    }
}

__global__ void k_add_finish(Ctl *c, unsigned long long count, unsigned long long C, double alpha,
                             const double *rank_cdf)
{
    if (threadIdx.x == 0 && blockIdx.x == 0) {
        fold_running_max(c, c->add_max_bits, alpha);
        c->add_max_bits = 0;
        c->cursor = (c->cursor + count) % C;
        const unsigned long long sz = c->size + count < C ? c->size + count : C;
        c->size = sz;
        if (rank_cdf) c->rank_total_bits = (unsigned long long)__double_as_longlong(rank_cdf[sz]);
    }
}

__global__ void k_fill(float *p, unsigned long long n, float v)
{
    for (unsigned long long i = blockIdx.x * (unsigned long long)blockDim.x + threadIdx.x; i < n;
         i += (unsigned long long)gridDim.x * blockDim.x)
        p[i] = v;
}

// ------------------------------------------------------------------------------------------
// Priority update for a few entries: the per-element propagation the post measures its level
// rebuild against ("Putting prioritized replay's segment tree on a GPU", Measuring the Trade
// Honestly: each changed leaf walks to the root).  One warp takes the entries in batch order;
// for each it writes the leaf, loads the sibling of every ancestor at once (lane l the sibling
// at height l) and recomputes the ancestors bottom-up, each the binary64 sum of its two
// children, lane l storing the node at height l + 1.  The warp orders its memory between
// entries, so a later entry sees an earlier one's nodes: the last writer wins and every node
// ends as the sum of its final children, as in a sequential update.
// ------------------------------------------------------------------------------------------
struct ElementArgs {
    TreeRefs t;
    Ctl *ctl;
    const long long *idx;
    const float *td;
    unsigned B;
    double alpha, eps;
    LeafPowAlpha lp;
};

__global__ void __launch_bounds__(32) k_upd_element(ElementArgs a)
{
    pdl_wait();
    pdl_release();
    const int lane = threadIdx.x;
    const TreeRefs t = a.t;
    const int D = t.D;
    const unsigned long long size = a.ctl->size;
    const float max_prev = __uint_as_float(a.ctl->max_raw_bits);
    unsigned batch_max = 0;
    bool bad = false;
    for (unsigned j0 = 0; j0 < a.B; j0 += 32) {
        const unsigned jl = j0 + lane;
        const long long iv = jl < a.B ? __ldg(a.idx + jl) : -1;
        const float tv = jl < a.B ? __ldg(a.td + jl) : 0.0f;
        const unsigned cnt = a.B - j0 < 32u ? a.B - j0 : 32u;
        for (unsigned q = 0; q < cnt; ++q) {
            const long long i = __shfl_sync(0xffffffffu, iv, (int)q);
            const float tq = __shfl_sync(0xffffffffu, tv, (int)q);
            if (i < 0 || (unsigned long long)i >= size) {
                bad = true;
                continue;
            }
            const float raw = td_to_raw(tq, a.eps, max_prev);
            batch_max = max(batch_max, __float_as_uint(raw));
            const float leaf = leaf_of(raw, a.lp);
            const unsigned long long v0 = t.n + (unsigned long long)i;
            double sv = 0.0;
            float sm = __int_as_float(0x7f800000);
            if (lane < D) {
                const unsigned long long sib = (v0 >> lane) ^ 1ull;
                sv = ld_sum_cg(t, sib);
                sm = ld_min_cg(t, sib);
            }
            if (lane == 0) t.L[i] = leaf;
            double v = (double)leaf, mine_v = 0.0;
            float m = leaf_min_value(leaf), mine_m = 0.0f;
            for (int l = 0; l < D; ++l) {
                v = v + __shfl_sync(0xffffffffu, sv, l);
                m = fmin_tree(m, __shfl_sync(0xffffffffu, sm, l));
                if (lane == l) {
                    mine_v = v;
                    mine_m = m;
                }
            }
            if (lane < D) {
                const unsigned long long node = v0 >> (lane + 1);
                t.S[node] = mine_v;
                t.M[node] = mine_m;
            }
            __syncwarp();
        }
    }
    if (lane == 0) {
        if (bad) atomicOr(&a.ctl->err_flags, kFlagBadIndex);
        fold_running_max(a.ctl, batch_max, a.alpha);
    }
}

// ------------------------------------------------------------------------------------------
// Priority update for batches that touch a large share of the slots ("Putting prioritized
// replay's segment tree on a GPU", Second Port and Measuring the Trade Honestly: the
// level-synchronous rebuild of every node costs O(k + n), the per-entry climb O(k log n), and
// the first wins once k is a large enough share of n).  The last writer wins through one
// winner word per slot: every valid entry j raises win[i] to j + 1 (atomicMax); the entry that
// then finds its own j + 1 there writes the slot and zeroes the word, so every word is zero
// again after the call without a clearing pass.  Proportional mode then rebuilds every level
// of both trees (k_rebuild_tree) and k_upd_finish folds the batch maximum.
// ------------------------------------------------------------------------------------------
struct ScatterArgs {
    TreeRefs t;
    float *raw_store;
    Ctl *ctl;
    DirtyRefs dirty;
    unsigned *win;
    const long long *idx;
    const float *td;
    unsigned B;
    double eps, alpha;
    LeafPowAlpha lp;
    int proportional;
    CrowdRefs crowd;   // hist non-null: count the entries per subtree
};

__global__ void __launch_bounds__(kThreads) k_upd_scatter(ScatterArgs a)
{
    pdl_wait();
    pdl_release();
    const unsigned long long size = a.ctl->size;
    const float max_prev = __uint_as_float(a.ctl->max_raw_bits);
    unsigned mymax = 0;
    int bad = 0;
    for (unsigned j = blockIdx.x * blockDim.x + threadIdx.x; j < a.B; j += gridDim.x * blockDim.x) {
        const long long i = __ldg(a.idx + j);
        if (i < 0 || (unsigned long long)i >= size) {
            bad = 1;
            continue;
        }
        mymax = max(mymax, __float_as_uint(td_to_raw(__ldg(a.td + j), a.eps, max_prev)));
        atomicMax(a.win + i, j + 1);
        if (a.crowd.hist) atomicAdd(a.crowd.hist + ((unsigned long long)i >> a.crowd.shift), 1u);
    }
    if (__syncthreads_or(bad) && threadIdx.x == 0) atomicOr(&a.ctl->err_flags, kFlagBadIndex);
    const unsigned bm = block_max_u32(mymax);
    if (threadIdx.x == 0 && bm) atomicMax(&a.ctl->batch_max_bits, bm);
}

__global__ void __launch_bounds__(kThreads) k_upd_apply(ScatterArgs a)
{
    pdl_wait();
    pdl_release();
    const unsigned long long size = a.ctl->size;
    const float max_prev = __uint_as_float(a.ctl->max_raw_bits);   // not folded until k_upd_finish
    for (unsigned j = blockIdx.x * blockDim.x + threadIdx.x; j < a.B; j += gridDim.x * blockDim.x) {
        const long long i = __ldg(a.idx + j);
        if (i < 0 || (unsigned long long)i >= size) continue;
        if (__ldcg(a.win + i) != j + 1) continue;   // a later entry holds this slot (or has taken it)
        a.win[i] = 0;
        const float raw = td_to_raw(__ldg(a.td + j), a.eps, max_prev);
        if (a.proportional) {
            a.t.L[i] = leaf_of(raw, a.lp);
        } else {
            const float old = a.raw_store[i];
            a.raw_store[i] = raw;
            mark_dirty(a.dirty, (unsigned long long)i, old);
        }
    }
}

// Batches of at most kBlockBatch entries without a tree to climb (rank and flat modes): one
// thread-block cluster of kBlockCtas CTAs does what k_upd_scatter, k_upd_apply and k_upd_finish
// do, in one launch (the random accesses of one batch, spread over kBlockCtas SMs rather than
// issued by one; hardware cluster barriers separate the phases).  Each thread keeps its entries in
// registers: it loads index and TD error, then at once raises the slot's winner word and (rank
// mode) reads the slot's raw priority and mark; after a cluster barrier, the entry that still
// finds its own position stores its priority and clears the word.  Rank mode marks each slot not
// yet marked in this epoch (the mark read before says which: this launch is the slot's only
// writer), with one counter increment per CTA for the list positions.  CTA 0 folds the batch
// maximum after a last cluster barrier.
constexpr int kBlockCtas = 8;
constexpr int kBlockThreads = 256;
constexpr int kBlockPer = 4;   // entries per thread, at most
constexpr unsigned kBlockBatch = (unsigned)(kBlockCtas * kBlockThreads * kBlockPer);   // 8192

__global__ void __launch_bounds__(kBlockThreads) k_upd_block(ScatterArgs a)
{
    __shared__ unsigned s_w[kBlockThreads / 32];
    // every CTA writes its count of new marks into every CTA's s_tot, and its batch maximum into
    // CTA 0's s_bmax (distributed shared memory, before the second cluster barrier)
    __shared__ unsigned s_tot[kBlockCtas], s_bmax[kBlockCtas];
    pdl_wait();
    pdl_release();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const unsigned crank = cluster_cta_rank();
    const unsigned gtid = crank * kBlockThreads + tid, gthreads = kBlockCtas * kBlockThreads;
    const unsigned long long size = a.ctl->size;
    const unsigned max_prev_bits = a.ctl->max_raw_bits;
    const float max_prev = __uint_as_float(max_prev_bits);
    const bool rank = !a.proportional;
    const unsigned epoch = rank && a.dirty.mark ? __ldcg(a.dirty.epoch) : 0u;
    // the list's length before this call: nothing else appends during it
    const unsigned count0 = rank && a.dirty.mark ? __ldcg(a.dirty.count) : 0u;
    constexpr unsigned kNone = 0xffffffffu;   // no entry, or an index outside the filled slots
    unsigned iv[kBlockPer];
    float tv[kBlockPer], oldv[kBlockPer];
    unsigned mword[kBlockPer];
#pragma unroll
    for (int u = 0; u < kBlockPer; ++u) {
        const unsigned j = gtid + u * gthreads;
        const long long i = j < a.B ? __ldg(a.idx + j) : -1;
        tv[u] = j < a.B ? __ldg(a.td + j) : 0.0f;
        iv[u] = (i < 0 || (unsigned long long)i >= size) ? kNone : (unsigned)i;
    }
    unsigned mymax = 0;
    int bad = 0;
#pragma unroll
    for (int u = 0; u < kBlockPer; ++u) {
        const unsigned j = gtid + u * gthreads;
        const unsigned i = iv[u];
        oldv[u] = 0.0f;
        mword[u] = 0u;
        if (j >= a.B) continue;
        if (i == kNone) {
            bad = 1;
            continue;
        }
        mymax = max(mymax, __float_as_uint(td_to_raw(tv[u], a.eps, max_prev)));
        atomicMax(a.win + i, j + 1);
        if (rank) {
            oldv[u] = a.raw_store[i];
            if (a.dirty.mark) mword[u] = a.dirty.mark[i];
        }
    }
    if (__syncthreads_or(bad) && tid == 0) atomicOr(&a.ctl->err_flags, kFlagBadIndex);
    cluster_sync_all();   // every winner word raised
    unsigned newmark = 0;   // bit u: entry u marks its slot for the first time
#pragma unroll
    for (int u = 0; u < kBlockPer; ++u) {
        const unsigned j = gtid + u * gthreads;
        const unsigned i = iv[u];
        if (i == kNone) continue;
        if (__ldcg(a.win + i) != j + 1) continue;   // a later entry holds this slot (or has taken it)
        a.win[i] = 0;
        const float raw = td_to_raw(tv[u], a.eps, max_prev);
        if (!rank) {
            a.t.L[i] = leaf_of(raw, a.lp);
        } else {
            a.raw_store[i] = raw;
            if (a.dirty.mark && mword[u] != epoch) {
                a.dirty.mark[i] = epoch;
                newmark |= 1u << u;
            }
        }
    }
    // this CTA's count of new marks (exclusive prefix over its threads) and batch maximum, to the
    // other CTAs; after the barrier each CTA places its marks after those of the CTAs before it
    unsigned inc = 0, c = 0;
    if (rank && a.dirty.mark) {
        c = __popc(newmark);
        inc = c;
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned x = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += x;
        }
        if (lane == 31) s_w[warp] = inc;
        __syncthreads();
    }
    unsigned before = 0, total = 0;
    if (rank && a.dirty.mark) {
        for (int w = 0; w < kBlockThreads / 32; ++w) {
            const unsigned x = s_w[w];
            if (w < warp) before += x;
            total += x;
        }
        __syncthreads();   // s_w is reused below
    }
    for (int o = 16; o > 0; o >>= 1) mymax = max(mymax, __shfl_xor_sync(0xffffffffu, mymax, o));
    if (lane == 0) s_w[warp] = mymax;
    __syncthreads();
    if (tid < kBlockCtas) st_cluster_u32(cluster_smem_addr(&s_tot[crank], (unsigned)tid), total);
    if (tid == 32) {
        unsigned bm = 0;
        for (int w = 0; w < kBlockThreads / 32; ++w) bm = max(bm, s_w[w]);
        st_cluster_u32(cluster_smem_addr(&s_bmax[crank], 0), bm);
    }
    cluster_sync_all();   // every CTA's count and maximum in
    if (rank && a.dirty.mark) {
        unsigned pos = count0 + before + inc - c;
        for (unsigned q = 0; q < crank; ++q) pos += s_tot[q];
#pragma unroll
        for (int u = 0; u < kBlockPer; ++u)
            if ((newmark >> u) & 1u) {
                if (pos < kMaxDirty) {
                    a.dirty.list[pos] = iv[u];
                    a.dirty.oldkey[pos] = order_key(oldv[u]);
                }
                ++pos;
            }
        if (crank == 0 && tid == 0) {
            unsigned all = 0;
            for (int q = 0; q < kBlockCtas; ++q) all += s_tot[q];
            *a.dirty.count = count0 + all;
        }
    }
    if (crank == 0 && tid == 32) {
        unsigned bm = 0;
        for (int q = 0; q < kBlockCtas; ++q) bm = max(bm, s_bmax[q]);
        if (bm > max_prev_bits) fold_running_max(a.ctl, bm, a.alpha);
    }
}

__global__ void k_upd_finish(Ctl *c, double alpha)
{
    pdl_wait();
    pdl_release();
    if (threadIdx.x == 0 && blockIdx.x == 0) {
        fold_running_max(c, c->batch_max_bits, alpha);
        c->batch_max_bits = 0;
    }
}

// ------------------------------------------------------------------------------------------
// Priority update: last-writer-wins scatter + dirty-ancestor upsweep, one launch.
// The tree below depth P is cut into 2^P subtrees and each subtree belongs to one warp (a CTA
// holds 4 or 16 of them), so nothing below depth P needs more than warp synchronisation:
//   1. every CTA reads the whole batch, coalesced (the first entries of each thread in flight
//      with the control words), and files each entry of its subtrees under the subtree's warp
//      (while the ring fills, the subtrees split only the part that holds filled slots);
//   2. each warp starts copying, for each of its entries, the siblings on the entry's path into
//      shared memory (cp.async, up to 16 levels), computes the entries' leaf values meanwhile,
//      sorts them by (leaf, batch position) -- in registers up to 32, in shared memory beyond --
//      keeps the last position of every leaf, and climbs its subtree 32 distinct leaves at a
//      time: joins of two paths are planned from one warp OR, and a chain of binary64 adds, one
//      height per loop iteration, carries nothing else;
//   3. the top: a grid of at most 16 CTAs runs as one cluster, and every warp writes its
//      subtree's root (and every CTA its batch maximum and most entries per subtree) into CTA
//      0's shared memory; after one cluster barrier CTA 0 builds the 2^P - 1 nodes above the
//      roots from there.  A larger grid uses an arrival ticket, and the last CTA reads the
//      roots back from L2.  The top CTA then rebuilds the spine above them while the ring
//      fills, and folds the batch maximum into the running maximum.
// A warp whose subtree receives more entries than its shared-memory list holds applies the
// batch in position order 32 entries at a time (later chunks overwrite earlier ones, so the
// last writer wins) and then rebuilds its whole subtree.
//
// Measured on GB300 (per-stage clock stamps, apex batch): the kernel is a chain of dependent
// steps in few warps, where each instruction of straight-line code costs about twice its warm
// time because it is fetched once per launch (a binary64 add alone takes 64 cycles); hence the
// loops over heights and levels rather than unrolled code, and no memory round trip left between
// the subtree climbs and the top (no fence, no reload of the roots).
// ------------------------------------------------------------------------------------------
// Two CTA shapes: 4 warps with lists of 512 entries (batches below 4096 entries), or 16 warps
// with lists of 128 (larger batches: a quarter as many CTAs read the whole batch, each in one
// round).  Both take the same list space; each warp has its own sibling prefetch area.
constexpr int kUpdMaxWarps = 16;
constexpr int kUpdMaxThreads = 32 * kUpdMaxWarps;
constexpr int kUpdSmallWarps = 4, kUpdSmallCap = 512;
constexpr int kUpdLargeWarps = 16, kUpdLargeCap = 128;
constexpr unsigned kUpdLargeBatch = 4096;
constexpr int kUpdWindow = 8;  // tree levels whose clean siblings load in one round

struct UpdArgs {
    TreeRefs t;
    float *raw_store;
    Ctl *ctl;
    DirtyRefs dirty;   // rank mode: slots written are marked for the next order merge
    const long long *idx;
    const float *td;
    unsigned B;
    int P;      // log2 number of subtrees
    int subs;   // subtrees per CTA (warps 0 .. subs-1 climb; all warps file the batch)
    int cap;    // entries a warp's list holds (more take the chunked path)
    int pb;     // bits for a batch position
    double alpha, eps;
    LeafPowAlpha lp;
    int proportional;
    int cluster;   // the grid is one thread-block cluster: CTA 0 builds the top after a cluster barrier
    unsigned *crowd_host;   // the most entries in one subtree goes here (host-mapped), or null
};

// One warp's entry lists in shared memory, `cap` entries each (36 bytes per entry).
struct WarpLists {
    unsigned long long *keys;  // (leaf offset << pb) | position
    unsigned *pay;             // entry slot carried through the sort
    float *rawv;               // raw priority by entry slot
    unsigned *ulist;           // distinct leaves, ascending (absolute)
    float *uraw;               // raw priority of each distinct leaf
};
constexpr size_t kListBytesPerEntry = 24;

__device__ __forceinline__ WarpLists warp_lists(unsigned char *smem, int w, int cap)
{
    unsigned char *b = smem + (size_t)w * kListBytesPerEntry * cap;
    WarpLists l;
    l.keys = reinterpret_cast<unsigned long long *>(b);
    b += 8 * (size_t)cap;
    l.pay = reinterpret_cast<unsigned *>(b);
    b += 4 * (size_t)cap;
    l.rawv = reinterpret_cast<float *>(b);
    b += 4 * (size_t)cap;
    l.ulist = reinterpret_cast<unsigned *>(b);
    b += 4 * (size_t)cap;
    l.uraw = reinterpret_cast<float *>(b);
    return l;
}

constexpr size_t kTopHeapBytes = (size_t)(2 << kMaxTopLog) * 12;  // the last CTA's top levels
constexpr size_t kListsBytes = kListBytesPerEntry * (kUpdSmallWarps * kUpdSmallCap > kUpdLargeWarps * kUpdLargeCap
                                                         ? kUpdSmallWarps * kUpdSmallCap : kUpdLargeWarps * kUpdLargeCap);
constexpr int kClusterRoots = 256;   // subtrees of a one-cluster grid: at most 16 CTAs of 16 warps

__device__ __forceinline__ void warp_bitonic_kv(unsigned long long *keys, unsigned *pay, int m2, int lane)
{
    for (int k = 2; k <= m2; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int t = lane; t < (m2 >> 1); t += 32) {
                const int i = ((t & ~(j - 1)) << 1) | (t & (j - 1));
                const int l = i + j;
                const bool up = (i & k) == 0;
                const unsigned long long ki = keys[i], kl = keys[l];
                if ((ki > kl) == up) {
                    keys[i] = kl;
                    keys[l] = ki;
                    const unsigned pi = pay[i];
                    pay[i] = pay[l];
                    pay[l] = pi;
                }
            }
            __syncwarp();
        }
    }
}

// Bitonic sort of one key per lane (ascending across lanes 0..31), carrying a payload.
// Bitonic sort of the keys of lanes [0, N) in each aligned group of N lanes (ascending), with a
// payload; lanes beyond the entries hold the largest key.
template <int N>
__device__ __forceinline__ void warp_sort_n(unsigned long long &key, unsigned &pay, int lane)
{
#pragma unroll
    for (int size = 2; size <= N; size <<= 1) {
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            const unsigned long long ok = __shfl_xor_sync(0xffffffffu, key, stride);
            const unsigned op = __shfl_xor_sync(0xffffffffu, pay, stride);
            const bool up = (lane & size) == 0;
            const bool lower = (lane & stride) == 0;
            const bool take = lower ? (up ? ok < key : ok > key) : (up ? ok > key : ok < key);
            if (take) {
                key = ok;
                pay = op;
            }
        }
    }
}

// The same for one 32-bit key per lane, without a payload (keys are distinct).
template <int N>
__device__ __forceinline__ void warp_sort_n32(unsigned &key, int lane)
{
#pragma unroll
    for (int size = 2; size <= N; size <<= 1) {
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            const unsigned ok = __shfl_xor_sync(0xffffffffu, key, stride);
            const bool up = (lane & size) == 0;
            const bool lower = (lane & stride) == 0;
            const bool take = lower ? (up ? ok < key : ok > key) : (up ? ok > key : ok < key);
            if (take) key = ok;
        }
    }
}

// Climb one warp's subtree when it has U <= 32 distinct leaves, one per lane, ascending: lane u
// holds local leaf li (leaf - base, base = the subtree's first leaf) and its leaf value.
//
// Let J be the height at which a lane's path joins the previous lane's (the bit length of the
// two local leaves' xor; lane 0 has none).  At height h the lane owns its node when h < J (or it
// is lane 0), and the owners of one height are in leaf order.  At a height where no lane has
// J = h + 1 no two owned nodes are siblings, so every owner adds its clean sibling.  At a height
// where some lane has J = h + 1 (a join), that lane's node is the right sibling of the node of the
// previous owner of the height: the previous owner adds the joining lane's value, taken by a
// shuffle, and the joining lane stops.  The joins are the set bits of one warp OR of 2^(J - 1), so
// the ballots and shuffles run at those heights only (at most U - 1 of them).
//
// The siblings were copied into the warp's prefetch area (prefetch_siblings) while the power and
// the sort ran: the chain of binary64 adds reads them from shared memory and carries nothing else.
// Each owner stores the node it computes; lane 0 ends with the subtree's root.
constexpr int kMaxClimb = 16;  // levels whose siblings are copied in the single prefetch round

struct ClimbLane {
    unsigned li;      // local leaf index
    int J;            // joining height with the previous lane (64: none)
    bool have;
    double vs;        // value of the lane's current node
    float vm;
};

// One level of the climb for heights beyond the prefetch round: children at height h, parent at
// h + 1.  `merge` is warp-uniform.
__device__ __forceinline__ void climb_level(const TreeRefs &t, unsigned long long top, int h, bool merge,
                                            int lane, ClimbLane &c, double sib_s, float sib_m)
{
    const bool own = c.have && (lane == 0 || c.J > h);
    const unsigned v = c.li >> h;
    bool compute = own;
    double ss = sib_s;
    float sm = sib_m;
    if (merge) {
        const unsigned own_h = __ballot_sync(0xffffffffu, own);
        const unsigned own_h1 = __ballot_sync(0xffffffffu, c.have && (lane == 0 || c.J > h + 1));
        const int R = __ffs(own_h & ~((2u << lane) - 1u)) - 1;   // next owner of height h
        const int src = R < 0 ? lane : R;
        const double e_s = __shfl_sync(0xffffffffu, c.vs, src);
        const float e_m = __shfl_sync(0xffffffffu, c.vm, src);
        if (v & 1u) {
            compute = own && (lane == 0 || c.J > h + 1);   // else the left sibling's owner adds
        } else if (R >= 0 && !((own_h1 >> R) & 1u)) {
            ss = e_s;                                       // the right sibling is dirty
            sm = e_m;
        }
    }
    if (compute) {
        c.vs = c.vs + ss;
        c.vm = fmin_tree(c.vm, sm);
        const unsigned long long node = (top >> (h + 1)) + (v >> 1);
        t.S[node] = c.vs;
        t.M[node] = c.vm;
    }
}

// A warp's sibling prefetch area in shared memory: for each of 32 slots, the siblings of a leaf's
// path at heights 1 .. kMaxClimb - 1 (S and M, height-major so that the 32 slots of one height are
// consecutive) and its sibling leaf.
struct SibArea {
    double *S;   // [kMaxClimb][32]
    float *M;    // [kMaxClimb][32]
    float *L;    // [32]
};
constexpr size_t kSibBytesPerWarp = (size_t)kMaxClimb * 32 * 8 + (size_t)kMaxClimb * 32 * 4 + 32 * 4;

// Dynamic shared memory of the update kernel: the entry lists (whose space the last CTA reuses for
// the top levels), then one prefetch area per warp.
static_assert(kTopHeapBytes <= kListsBytes, "top levels reuse the lists");
constexpr size_t update_smem_bytes(int warps) { return kListsBytes + (size_t)warps * kSibBytesPerWarp; }

__device__ __forceinline__ SibArea sib_area(unsigned char *base, int w)
{
    unsigned char *b = base + (size_t)w * kSibBytesPerWarp;
    SibArea s;
    s.S = reinterpret_cast<double *>(b);
    s.M = reinterpret_cast<float *>(b + (size_t)kMaxClimb * 32 * 8);
    s.L = s.M + kMaxClimb * 32;
    return s;
}

__device__ __forceinline__ void cp_async4(void *smem, const void *gmem)
{
    const unsigned sa = (unsigned)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(sa), "l"(gmem) : "memory");
}

__device__ __forceinline__ void cp_async8(void *smem, const void *gmem)
{
    const unsigned sa = (unsigned)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(sa), "l"(gmem) : "memory");
}

// Waits for this thread's copies; the warp barrier then makes every lane's copies visible to the
// whole warp.
__device__ __forceinline__ void cp_async_wait_warp()
{
    asm volatile("cp.async.wait_all;" ::: "memory");
    __syncwarp();
}

// Starts the copies (no wait) of the siblings on the path of leaf node v0 (= n + leaf) at
// heights 0 .. hpre - 1 into slot `slot` of the area.
__device__ __forceinline__ void prefetch_siblings(const TreeRefs &t, unsigned long long v0, int hpre,
                                                  const SibArea &p, int slot)
{
    cp_async4(p.L + slot, t.L + ((v0 ^ 1ull) - t.n));
#pragma unroll 1
    for (int h = 1; h < hpre; ++h) {
        const unsigned long long sib = (v0 >> h) ^ 1ull;
        cp_async8(p.S + h * 32 + slot, t.S + sib);
        cp_async4(p.M + h * 32 + slot, t.M + sib);
    }
}

// The climb (see above).  Lane u < U: local leaf li, leaf value lv, siblings complete in slot
// `slot` of the area.  Writes the leaves and every recomputed node; lane 0 returns the subtree's
// root (height `shift`) in *rs / *rm.
template <int W>
__device__ void warp_climb(const TreeRefs &t, int U, int shift, int lane, unsigned long long base,
                           unsigned li, float lv, const SibArea &p, int slot, double *rs, float *rm)
{
    constexpr unsigned kAll = 0xffffffffu;
    ClimbLane c;
    c.li = li;
    c.have = lane < U;
    const unsigned prev = __shfl_up_sync(kAll, li, 1);
    c.J = (c.have && lane > 0) ? 32 - __clz(prev ^ li) : 64;
    const unsigned long long v0 = t.n + base + li;
    const int hpre = min(shift, kMaxClimb);
    c.vs = 0.0;
    c.vm = 0.0f;
    if (c.have) {
        t.L[base + li] = lv;
        c.vs = (double)lv;
        c.vm = leaf_min_value(lv);
    }
    const unsigned joins = __reduce_or_sync(kAll, (c.have && lane > 0 && c.J <= hpre) ? 1u << (c.J - 1) : 0u);
    const unsigned above = ~((2u << lane) - 1u);
    const float kInf = __int_as_float(0x7f800000);
    // The chain, one height per iteration: run once per launch, a loop's few instructions are
    // fetched once where unrolled heights would each be fetched (measured on GB300: about half the
    // time per height).  A lane that does not add at a height adds +0 and takes the minimum with
    // +inf (every value is >= +0); the next height's sibling is read while this one is added.
    float lsib = p.L[slot];
    double ns = (double)lsib;
    float nm = leaf_min_value(lsib);
#pragma unroll 1
    for (int h = 0; h < hpre; ++h) {
        double as = ns;
        float am = nm;
        if (h + 1 < hpre) {
            ns = p.S[(h + 1) * 32 + slot];
            nm = p.M[(h + 1) * 32 + slot];
        }
        const bool own = c.have && (lane == 0 || c.J > h);
        bool add = own;
        if ((joins >> h) & 1u) {
            const bool right = own && lane > 0 && c.J == h + 1;   // joins the previous owner at h + 1
            const unsigned ob = __ballot_sync(kAll, own);
            const unsigned rb = __ballot_sync(kAll, right);
            const int R = __ffs(ob & above) - 1;                // next owner of height h
            const int src = R < 0 ? lane : R;
            const double e = __shfl_sync(kAll, c.vs, src);
            const float em = __shfl_sync(kAll, c.vm, src);
            if (own && R >= 0 && ((rb >> R) & 1u)) {
                as = e;
                am = em;
            }
            add = own && !right;
        }
        c.vs = c.vs + (add ? as : 0.0);
        c.vm = fmin_tree(c.vm, add ? am : kInf);
        if (add) {
            const unsigned long long node = v0 >> (h + 1);
            t.S[node] = c.vs;
            t.M[node] = c.vm;
        }
    }
    // heights beyond the prefetch round (subtrees deeper than kMaxClimb levels), W per round
    const unsigned long long top = t.n + base;
    for (int h0 = hpre; h0 < shift; h0 += W) {
        double qs[W];
        float qm[W];
#pragma unroll
        for (int w = 0; w < W; ++w) {
            const int h = h0 + w;
            qs[w] = 0.0;
            qm[w] = 0.0f;
            if (c.have && h < shift && (lane == 0 || c.J > h)) {
                const unsigned long long sib = (top >> h) + ((li >> h) ^ 1u);
                qs[w] = t.S[sib];
                qm[w] = t.M[sib];
            }
        }
#pragma unroll
        for (int w = 0; w < W; ++w) {
            const int h = h0 + w;
            const bool merge = __any_sync(kAll, c.have && lane > 0 && c.J == h + 1);
            if (h < shift) climb_level(t, top, h, merge, lane, c, qs[w], qm[w]);
        }
    }
    *rs = c.vs;
    *rm = c.vm;
}

// Files the batch entries of this CTA's subtrees under their warp's list (slot order is the
// order of arrival; the sort below restores batch order).  Thread t takes entries t + u blockDim,
// U at a time; the first U arrive preloaded.  Returns this thread's largest raw priority among the
// filed entries.
template <int U>
__device__ __forceinline__ void load_entries(const UpdArgs &a, unsigned j0, long long (&iv)[U], float (&tv)[U])
{
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const unsigned j = j0 + u * blockDim.x;
        iv[u] = j < a.B ? __ldg(a.idx + j) : -2;
        tv[u] = j < a.B ? __ldg(a.td + j) : 0.0f;
    }
}

template <int U>
__device__ __forceinline__ unsigned file_batch(const UpdArgs &a, unsigned char *lists, int *s_cnt,
                                               unsigned long long first_sub, int shift,
                                               unsigned long long size, float max_prev,
                                               long long (&iv)[U], float (&tv)[U])
{
    unsigned mymax = 0;
    for (unsigned j0 = threadIdx.x; j0 < a.B; j0 += U * blockDim.x) {
        if (j0 != threadIdx.x) load_entries<U>(a, j0, iv, tv);
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const unsigned j = j0 + u * blockDim.x;
            const long long i = iv[u];
            if (i == -2) continue;
            if (i < 0 || (unsigned long long)i >= size) {
                if (blockIdx.x == 0) atomicOr(&a.ctl->err_flags, kFlagBadIndex);
                continue;
            }
            const unsigned long long sub = (unsigned long long)i >> shift;
            if (sub < first_sub || sub >= first_sub + a.subs) continue;
            const int w = (int)(sub - first_sub);
            const float raw = td_to_raw(tv[u], a.eps, max_prev);
            mymax = max(mymax, __float_as_uint(raw));
            const int slot = atomicAdd(&s_cnt[w], 1);
            if (slot < a.cap) {
                const WarpLists wl = warp_lists(lists, w, a.cap);
                wl.keys[slot] = (((unsigned long long)i - (sub << shift)) << a.pb) | j;
                wl.pay[slot] = (unsigned)slot;
                wl.rawv[slot] = raw;
            }
        }
    }
    return mymax;
}

template <int W>
__global__ void __launch_bounds__(kUpdMaxThreads) k_update(UpdArgs a)
{
    extern __shared__ __align__(16) unsigned char smem_raw[];
    unsigned char *lists = smem_raw;
    unsigned char *sibs = smem_raw + kListsBytes;   // the warps' sibling prefetch areas
    __shared__ int s_cnt[kUpdMaxWarps];
    __shared__ unsigned s_max;
    __shared__ LeafPowTables s_lp;
    // one-cluster grids: CTA 0 receives every subtree's root and every CTA's batch maximum and
    // most entries per subtree here (distributed shared memory), one slot per writer
    __shared__ double s_rootS[2 * kClusterRoots];   // a heap: the roots at [2^P, 2^(P+1))
    __shared__ float s_rootM[2 * kClusterRoots];
    __shared__ unsigned s_cbmax[16], s_ccnt[16];
    {   // the power's tables (constant since the library loaded), staged while the batch is read
        const unsigned *src = reinterpret_cast<const unsigned *>(&g_leafpow);
        unsigned *dst = reinterpret_cast<unsigned *>(&s_lp);
        for (int i = threadIdx.x; i < (int)(sizeof(LeafPowTables) / 4); i += blockDim.x) dst[i] = src[i];
    }
    // first half of a cluster barrier: the second half, before the first write into CTA 0's
    // shared memory, ensures every CTA of the cluster has started
    if (a.cluster) cluster_arrive_relaxed();
    pdl_wait();
    pdl_release();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int D = a.t.D;
    const unsigned long long n = a.t.n;
    const unsigned long long size = a.ctl->size;
    // While the ring fills, every valid index lies below `size`.  The 2^P subtrees are then
    // taken at depth P + skip, the subtree of node 2^skip split in 2^P, where skip is the
    // largest such that [0, n >> skip) still holds [0, size): the batch spreads over every warp
    // instead of the few whose subtrees hold the filled slots.  Nodes above depth skip off the
    // left spine cover only unused slots; the spine is rebuilt at the end.
    int skip = 0;
    while (a.P + skip + 1 <= D - 1 && size <= (n >> (skip + 1))) ++skip;
    const int shift = D - a.P - skip;
    const unsigned long long nsub = 1ull << a.P;
    const unsigned long long first_sub = (unsigned long long)blockIdx.x * a.subs;
    // the first U entries of this thread (indices and TD errors), in flight with the control words
    const unsigned per_round = (a.B + blockDim.x - 1) / blockDim.x;
    long long iv4[4], iv8[8], iv16[16];
    float tv4[4], tv8[8], tv16[16];
    if (per_round <= 4) load_entries<4>(a, tid, iv4, tv4);
    else if (per_round <= 8) load_entries<8>(a, tid, iv8, tv8);
    else load_entries<16>(a, tid, iv16, tv16);
    const unsigned max_prev_bits = a.ctl->max_raw_bits;
    const float max_prev = __uint_as_float(max_prev_bits);
    // the crowding report's sequence number, taken now so that the top CTA does not wait for it
    // (the top CTA's report, the maximum's fold and the resets run on a thread of warp 1, beside
    // warp 0's rebuild of the top levels)
    const int reporter = blockDim.x > 32 ? 32 : 0;
    unsigned crowd_seq = 0;
    if (a.cluster && a.crowd_host && blockIdx.x == 0 && tid == reporter) crowd_seq = atomicAdd(&a.ctl->crowd_seq, 1u);
    if (tid < kUpdMaxWarps) s_cnt[tid] = 0;
    if (tid == 0) s_max = 0;
    __syncthreads();

    // 1. file this CTA's entries under their subtree's warp (every CTA reads the whole batch:
    //    indices and TD errors together, 4, 8 or 16 per thread in flight as the batch grows)
    unsigned mymax = 0;
    if (per_round <= 4) mymax = file_batch<4>(a, lists, s_cnt, first_sub, shift, size, max_prev, iv4, tv4);
    else if (per_round <= 8) mymax = file_batch<8>(a, lists, s_cnt, first_sub, shift, size, max_prev, iv8, tv8);
    else mymax = file_batch<16>(a, lists, s_cnt, first_sub, shift, size, max_prev, iv16, tv16);
    for (int o = 16; o > 0; o >>= 1) mymax = max(mymax, __shfl_xor_sync(0xffffffffu, mymax, o));
    if (lane == 0 && mymax) atomicMax(&s_max, mymax);
    __syncthreads();
    if (!a.cluster && tid == 0 && s_max) atomicMax(&a.ctl->batch_max_bits, s_max);
    if (!a.cluster && tid == 0 && a.crowd_host) {   // crowding: the most entries one of this CTA's subtrees received
        int m = 0;
        for (int w = 0; w < a.subs; ++w) m = max(m, s_cnt[w]);
        if (m) atomicMax(&a.ctl->crowd_max, (unsigned)m);
    }

    // 2. one warp per subtree
    const unsigned long long sub = first_sub + warp;
    const int m = s_cnt[warp];
    const bool has_sub = warp < a.subs && sub < nsub;
    const unsigned long long root = (n + (sub << shift)) >> shift;   // the subtree's root node
    double root_s = 0.0;   // lane 0: the subtree root's value once this warp is done
    float root_m = 0.0f;
    if (a.proportional && has_sub && m == 0 && lane == 0) {   // untouched: as stored
        root_s = a.t.S[root];
        root_m = a.t.M[root];
    }
    if (has_sub && m > 0) {
        const WarpLists wl = warp_lists(lists, warp, a.cap);
        const unsigned long long base = sub << shift;
        if (m > a.cap) {
            for (unsigned p0 = 0; p0 < a.B; p0 += 32) {
                const unsigned j = p0 + lane;
                long long i = -1;
                if (j < a.B) i = __ldg(a.idx + j);
                const bool mine = i >= 0 && (unsigned long long)i < size && ((unsigned long long)i >> shift) == sub;
                const unsigned long long key = mine ? (unsigned long long)i : ~0ull;
                const unsigned peers = __match_any_sync(0xffffffffu, key);
                if (mine && (31 - __clz(peers)) == lane) {  // the last lane of this chunk for the leaf
                    const float raw = td_to_raw(__ldg(a.td + j), a.eps, max_prev);
                    if (a.proportional) a.t.L[i] = leaf_of(raw, a.lp);
                    else {
                        const float old = a.raw_store[i];
                        a.raw_store[i] = raw;
                        mark_dirty(a.dirty, (unsigned long long)i, old);
                    }
                }
                __syncwarp();
            }
            if (a.proportional) {
                for (int h = 1; h <= shift; ++h) {
                    const unsigned long long cnt = 1ull << (shift - h);
                    const unsigned long long first = (n + base) >> h;
                    for (unsigned long long q = lane; q < cnt; q += 32) {
                        const unsigned long long node = first + q;
                        a.t.S[node] = ld_sum(a.t, 2 * node) + ld_sum(a.t, 2 * node + 1);
                        a.t.M[node] = fmin_tree(ld_min(a.t, 2 * node), ld_min(a.t, 2 * node + 1));
                    }
                    __syncwarp();
                }
                if (lane == 0) {   // lane 0 computed the root last
                    root_s = a.t.S[root];
                    root_m = a.t.M[root];
                }
            }
        } else if (m <= 32) {
            // one entry per lane (entry l of the list on lane l): the copies of its path's
            // siblings start and its leaf value is computed, then the entries are sorted in
            // registers, the last position of each leaf kept, and the u-th surviving leaf moved to
            // lane u, which climbs with the siblings its entry's lane copied
            const bool have = lane < m;
            unsigned long long key = have ? wl.keys[lane] : ~0ull;
            const float raw_e = have ? wl.rawv[lane] : 0.0f;   // pay[l] = l before the sort
            const SibArea sp = sib_area(sibs, warp);
            float lv_e = 0.0f;
            // entries of the same leaf share one copy of its path's siblings: the lowest lane of
            // each such group copies them into its slot
            const unsigned same = __match_any_sync(0xffffffffu, have ? (unsigned)(key >> a.pb) : 0xffffffffu);
            const int copier = __ffs(same) - 1;
            if (a.proportional && have) {
                if (copier == lane) prefetch_siblings(a.t, n + base + (key >> a.pb), min(shift, kMaxClimb), sp, lane);
                lv_e = leaf_of(raw_e, a.lp, s_lp);
            }
            // the sort key (leaf, batch position) with the list position beside it: one 32-bit
            // word when the three fit (then the position travels in the low 5 bits), else 64 bits
            // with a payload
            unsigned li, U;
            int slot;
            if (shift + a.pb + 5 <= 32) {
                unsigned k32 = have ? ((unsigned)key << 5) | (unsigned)lane : ~0u;
                if (m <= 8) warp_sort_n32<8>(k32, lane);
                else if (m <= 16) warp_sort_n32<16>(k32, lane);
                else warp_sort_n32<32>(k32, lane);
                const unsigned sh = a.pb + 5;
                const unsigned nxt = __shfl_down_sync(0xffffffffu, k32, 1);
                const bool win = lane < m && (lane == m - 1 || (nxt >> sh) != (k32 >> sh));
                const unsigned bal = __ballot_sync(0xffffffffu, win);
                U = __popc(bal);
                const int from = lane < (int)U ? (int)__fns(bal, 0, lane + 1) : 0;
                const unsigned k_from = __shfl_sync(0xffffffffu, k32, from);
                li = k_from >> sh;
                slot = (int)(k_from & 31u);
            } else {
                unsigned pay = lane;
                if (m <= 8) warp_sort_n<8>(key, pay, lane);
                else if (m <= 16) warp_sort_n<16>(key, pay, lane);
                else warp_sort_n<32>(key, pay, lane);
                const unsigned long long nxt = __shfl_down_sync(0xffffffffu, key, 1);
                const bool win = lane < m && (lane == m - 1 || (nxt >> a.pb) != (key >> a.pb));
                const unsigned bal = __ballot_sync(0xffffffffu, win);
                U = __popc(bal);
                const int from = lane < (int)U ? (int)__fns(bal, 0, lane + 1) : 0;
                const unsigned long long k_from = __shfl_sync(0xffffffffu, key, from);
                slot = (int)__shfl_sync(0xffffffffu, pay, from);   // the entry's list position
                li = (unsigned)(k_from >> a.pb);                    // local leaf index
            }
            const float raw = __shfl_sync(0xffffffffu, raw_e, slot);
            const float lv = __shfl_sync(0xffffffffu, lv_e, slot);
            const int cslot = __shfl_sync(0xffffffffu, copier, slot);   // where the leaf's siblings are
            if (a.proportional) {
                cp_async_wait_warp();
                warp_climb<W>(a.t, (int)U, shift, lane, base, lane < (int)U ? li : 0u, lv, sp,
                              lane < (int)U ? cslot : 0, &root_s, &root_m);
            } else if (lane < (int)U) {
                const float old = a.raw_store[base + li];
                a.raw_store[base + li] = raw;
                mark_dirty(a.dirty, base + li, old);
            }
        } else {
            int m2 = 2;
            while (m2 < m) m2 <<= 1;
            for (int i = m + lane; i < m2; i += 32) wl.keys[i] = ~0ull;
            __syncwarp();
            warp_bitonic_kv(wl.keys, wl.pay, m2, lane);
            // distinct leaves, keeping the last batch position of each; compacted in order
            int U = 0;
            for (int k0 = 0; k0 < m; k0 += 32) {
                const int k = k0 + lane;
                bool win = false;
                if (k < m) win = (k == m - 1) || ((wl.keys[k + 1] >> a.pb) != (wl.keys[k] >> a.pb));
                const unsigned bal = __ballot_sync(0xffffffffu, win);
                const int u = U + __popc(bal & ((1u << lane) - 1u));
                unsigned long long leaf = 0;
                float raw = 0.0f;
                if (win) {
                    leaf = base + (wl.keys[k] >> a.pb);
                    raw = wl.rawv[wl.pay[k]];
                }
                __syncwarp();
                if (win) {
                    wl.ulist[u] = (unsigned)leaf;
                    if (a.proportional) {
                        wl.uraw[u] = raw;
                    } else {
                        const float old = a.raw_store[leaf];
                        a.raw_store[leaf] = raw;
                        mark_dirty(a.dirty, leaf, old);
                    }
                }
                U += __popc(bal);
            }
            __syncwarp();
            if (a.proportional) {
                // 32 distinct leaves at a time in ascending order, each group after the previous
                // one has stored its nodes: a later group reads the earlier groups' nodes as its
                // siblings and rewrites the ancestors they share
                const SibArea sp = sib_area(sibs, warp);
                for (int c0 = 0; c0 < U; c0 += 32) {
                    const int Uc = min(32, U - c0);
                    const bool have = lane < Uc;
                    const unsigned li = have ? wl.ulist[c0 + lane] - (unsigned)base : 0u;
                    float lv = 0.0f;
                    if (have) {
                        prefetch_siblings(a.t, n + base + li, min(shift, kMaxClimb), sp, lane);
                        lv = leaf_of(wl.uraw[c0 + lane], a.lp, s_lp);
                    }
                    cp_async_wait_warp();
                    warp_climb<W>(a.t, Uc, shift, lane, base, li, lv, sp, lane, &root_s, &root_m);
                    __syncwarp();
                }
            }
        }
    }

    // 3. the levels above this CTA's 2^lg subtrees that no other CTA reaches, from the warps'
    //    roots in shared memory (the CTA's group ends in one node of depth P + skip - lg); then
    //    the last CTA rebuilds the top Pt = P - lg levels and folds in the batch maximum (when the
    //    grid is one cluster: CTA 0, after a cluster barrier, without the arrival ticket)
    int lg = 0;
    while ((1 << (lg + 1)) <= a.subs && lg + 1 <= a.P) ++lg;
    const int Pt = a.P - lg;
    if (a.proportional && lg > 0) {
        __shared__ double s_gS[kUpdMaxWarps];
        __shared__ float s_gM[kUpdMaxWarps];
        if (lane == 0 && warp < (1 << lg)) {
            s_gS[warp] = root_s;
            s_gM[warp] = root_m;
        }
        __syncthreads();
        if (warp == 0) {
            double gs = 0.0;
            float gm = 0.0f;
#pragma unroll 1
            for (int l = 1; l <= lg; ++l) {
                const int cnt = 1 << (lg - l);
                if (lane < cnt) {
                    gs = s_gS[2 * lane] + s_gS[2 * lane + 1];
                    gm = fmin_tree(s_gM[2 * lane], s_gM[2 * lane + 1]);
                    const unsigned long long node = (1ull << (a.P + skip - l)) + (first_sub >> l) + lane;
                    a.t.S[node] = gs;
                    a.t.M[node] = gm;
                }
                __syncwarp();
                if (lane < cnt) {
                    s_gS[lane] = gs;
                    s_gM[lane] = gm;
                }
                __syncwarp();
            }
            root_s = gs;   // lane 0: the group's node
            root_m = gm;
        }
    }
    bool top;
    if (a.cluster) {
        // every group's node and this CTA's maxima to CTA 0; the barrier's release and acquire
        // order them (and every node stored above) before CTA 0's reads
        cluster_wait_acquire();
        if (a.proportional && lane == 0 && (lg > 0 ? warp == 0 : has_sub)) {
            const unsigned hi = (1u << Pt) + (unsigned)(lg > 0 ? blockIdx.x : sub);
            st_cluster_f64(cluster_smem_addr(&s_rootS[hi], 0), root_s);
            st_cluster_f32(cluster_smem_addr(&s_rootM[hi], 0), root_m);
        }
        if (tid == 0) {
            int mc = 0;
            for (int w = 0; w < a.subs; ++w) mc = max(mc, s_cnt[w]);
            st_cluster_u32(cluster_smem_addr(&s_cbmax[blockIdx.x], 0), s_max);
            st_cluster_u32(cluster_smem_addr(&s_ccnt[blockIdx.x], 0), (unsigned)mc);
        }
        cluster_sync_all();
        top = blockIdx.x == 0;
    } else {
        top = last_to_arrive(&a.ctl->ticket_update);
    }
    if (top && tid == reporter) {
        Ctl *cc = a.ctl;
        if (a.cluster) {
            // the CTAs' counts and maxima gathered here; the running maximum and the report's
            // sequence number read at the start
            if (a.crowd_host) {   // every CTA's count is in: to the host
                unsigned mc = 0;
                for (unsigned c = 0; c < gridDim.x; ++c) mc = max(mc, s_ccnt[c]);
                *(volatile unsigned *)a.crowd_host = crowd_word(a.P, crowd_seq, mc);
            }
            unsigned bm = 0;
            for (unsigned c = 0; c < gridDim.x; ++c) bm = max(bm, s_cbmax[c]);
            if (bm > max_prev_bits) fold_running_max(cc, bm, a.alpha);
        } else {
            // the count, the sequence number and the batch maximum requested together (one
            // round trip), then the report, the fold and the resets
            const unsigned mc = a.crowd_host ? atomicExch(&cc->crowd_max, 0u) : 0u;
            const unsigned seq = a.crowd_host ? atomicAdd(&cc->crowd_seq, 1u) : 0u;
            const unsigned bm = __ldcg(&cc->batch_max_bits);
            if (a.crowd_host) *(volatile unsigned *)a.crowd_host = crowd_word(a.P, seq, mc);
            if (bm > max_prev_bits) fold_running_max(cc, bm, a.alpha);
            cc->batch_max_bits = 0;
            cc->ticket_update = 0;
        }
    }
    if (top) {
        if (a.cluster && a.proportional) {
            // warp 0: the levels above the groups' nodes in the shared-memory heap, one level per
            // iteration (nodes of depth l + skip stored as they are made)
            if (warp == 0) {
#pragma unroll 1
                for (int l = Pt - 1; l >= 0; --l) {
                    const int lw = 1 << l;
                    for (int i = lane; i < lw; i += 32) {
                        const int node = lw + i;
                        const double sum = s_rootS[2 * node] + s_rootS[2 * node + 1];
                        const float mn = fmin_tree(s_rootM[2 * node], s_rootM[2 * node + 1]);
                        s_rootS[node] = sum;
                        s_rootM[node] = mn;
                        a.t.S[((unsigned long long)lw << skip) + i] = sum;
                        a.t.M[((unsigned long long)lw << skip) + i] = mn;
                    }
                    __syncwarp();
                }
            }
        } else if (a.proportional && Pt > 0 && Pt <= 8) {
            // warp 0: lane l first combines its g = 2^(P-5) depth-P nodes (P >= 5) down to one
            // node of depth 5 in registers, or starts from depth-P node l (P < 5); every level
            // above is one shuffle and one add
            if (warp == 0) {
                const int P = Pt;
                double sv = 0.0;
                float mv = __int_as_float(0x7f800000);
                int w;   // nodes of the current depth, held by lanes 0, st, 2 st, ...
                if (P >= 5) {
                    const int g = 1 << (P - 5);
                    double gs[8];
                    float gm[8];
                    const unsigned long long c0 = (1ull << (P + skip)) + (unsigned long long)lane * g;
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        gs[i] = i < g ? ld_sum_cg(a.t, c0 + i) : 0.0;
                        gm[i] = i < g ? ld_min_cg(a.t, c0 + i) : 0.0f;
                    }
#pragma unroll
                    for (int half = 4; half >= 1; half >>= 1) {
                        if (2 * half <= g) {
#pragma unroll
                            for (int i = 0; i < half; ++i) {
                                gs[i] = gs[2 * i] + gs[2 * i + 1];
                                gm[i] = fmin_tree(gm[2 * i], gm[2 * i + 1]);
                            }
                            // the sums are this lane's nodes of depth 5 + log2(half)
                            const int dlev = 5 + (31 - __clz(half));
#pragma unroll
                            for (int i = 0; i < half; ++i) {
                                const unsigned long long node = (1ull << (dlev + skip)) + (unsigned long long)lane * half + i;
                                a.t.S[node] = gs[i];
                                a.t.M[node] = gm[i];
                            }
                        }
                    }
                    sv = gs[0];   // depth-(5 + skip) node 32 * 2^skip + lane
                    mv = gm[0];
                    w = 32;
                } else {
                    w = 1 << P;
                    if (lane < w) {
                        sv = ld_sum_cg(a.t, ((unsigned long long)w << skip) + lane);
                        mv = ld_min_cg(a.t, ((unsigned long long)w << skip) + lane);
                    }
                }
                for (int st = 1; w > 1; st <<= 1, w >>= 1) {
                    const double os = __shfl_down_sync(0xffffffffu, sv, st);
                    const float om = __shfl_down_sync(0xffffffffu, mv, st);
                    if ((lane & (2 * st - 1)) == 0 && lane < w * st) {
                        sv = sv + os;
                        mv = fmin_tree(mv, om);
                        const unsigned long long node = ((unsigned long long)(w >> 1) << skip) + lane / (2 * st);
                        a.t.S[node] = sv;
                        a.t.M[node] = mv;
                    }
                }
            }
        } else if (a.proportional && Pt >= 7 && Pt <= 10 && (blockDim.x >> 5) >= 4) {
            // four warps: warp w rebuilds the subtree of node 4 + w from its 2^(P-2) depth-P
            // nodes (g = 2^(P-7) per lane combined in registers down to depth 7, then five
            // shuffle levels down to depth 2); warp 0 then adds nodes 4..7 up to the root
            __shared__ double s_q[4];
            __shared__ float s_qm[4];
            const int P = Pt;
            const int g = 1 << (P - 7);
            if (warp < 4) {
            double gs[8];
            float gm[8];
            const unsigned long long c0 = (1ull << (P + skip)) + ((unsigned long long)warp << (P - 2)) + (unsigned long long)lane * g;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                gs[i] = i < g ? ld_sum_cg(a.t, c0 + i) : 0.0;
                gm[i] = i < g ? ld_min_cg(a.t, c0 + i) : 0.0f;
            }
#pragma unroll
            for (int half = 4; half >= 1; half >>= 1) {
                if (2 * half <= g) {
#pragma unroll
                    for (int i = 0; i < half; ++i) {
                        gs[i] = gs[2 * i] + gs[2 * i + 1];
                        gm[i] = fmin_tree(gm[2 * i], gm[2 * i + 1]);
                    }
                    const int dlev = 7 + (31 - __clz(half));   // depth of these sums
#pragma unroll
                    for (int i = 0; i < half; ++i) {
                        const unsigned long long node = (1ull << (dlev + skip)) + ((unsigned long long)warp << (dlev - 2)) +
                                                        (unsigned long long)lane * half + i;
                        a.t.S[node] = gs[i];
                        a.t.M[node] = gm[i];
                    }
                }
            }
            double sv = gs[0];   // depth-7 node 128 + 32 warp + lane
            float mv = gm[0];
            for (int st = 1, w = 32, dep = 7; w > 1; st <<= 1, w >>= 1, --dep) {
                const double os = __shfl_down_sync(0xffffffffu, sv, st);
                const float om = __shfl_down_sync(0xffffffffu, mv, st);
                if ((lane & (2 * st - 1)) == 0) {
                    sv = sv + os;
                    mv = fmin_tree(mv, om);
                    const unsigned long long node = (1ull << (dep - 1 + skip)) + ((unsigned long long)warp << (dep - 3)) +
                                                    lane / (2 * st);
                    a.t.S[node] = sv;
                    a.t.M[node] = mv;
                }
            }
            if (lane == 0) {
                s_q[warp] = sv;
                s_qm[warp] = mv;
            }
            }   // warp < 4
            __syncthreads();
            if (warp == 0) {
                double qv = lane < 4 ? s_q[lane] : 0.0;   // nodes 4..7 on lanes 0..3
                float qm = lane < 4 ? s_qm[lane] : __int_as_float(0x7f800000);
                for (int st = 1, w = 4; w > 1; st <<= 1, w >>= 1) {
                    const double os = __shfl_down_sync(0xffffffffu, qv, st);
                    const float om = __shfl_down_sync(0xffffffffu, qm, st);
                    if ((lane & (2 * st - 1)) == 0 && lane < w * st) {
                        qv = qv + os;
                        qm = fmin_tree(qm, om);
                        const unsigned long long node = ((unsigned long long)(w >> 1) << skip) + lane / (2 * st);
                        a.t.S[node] = qv;
                        a.t.M[node] = qm;
                    }
                }
            }
        } else if (a.proportional && Pt > 0) {
            double *heapS = reinterpret_cast<double *>(smem_raw);
            float *heapM = reinterpret_cast<float *>(heapS + (2 << kMaxTopLog));
            const int P = Pt;
            const int width = 1 << P;
            for (int i = tid; i < width; i += blockDim.x) {
                heapS[width + i] = ld_sum_cg(a.t, ((unsigned long long)width << skip) + i);
                heapM[width + i] = ld_min_cg(a.t, ((unsigned long long)width << skip) + i);
            }
            for (int l = P - 1; l >= 0; --l) {
                __syncthreads();
                const int lw = 1 << l;
                for (int i = tid; i < lw; i += blockDim.x) {
                    const int node = lw + i;
                    const double sum = heapS[2 * node] + heapS[2 * node + 1];
                    const float mn = fmin_tree(heapM[2 * node], heapM[2 * node + 1]);
                    heapS[node] = sum;
                    heapM[node] = mn;
                    a.t.S[((unsigned long long)lw << skip) + i] = sum;
                    a.t.M[((unsigned long long)lw << skip) + i] = mn;
                }
            }
        }
        if (a.proportional && skip > 0) {
            // the left spine from node 2^skip (rebuilt above, or the single subtree's root) up to
            // the root; each right sibling on it covers slots at or beyond n >> skip, untouched
            __syncthreads();
            if (tid == 0) {
                double sv = ld_sum_cg(a.t, 1ull << skip);
                float mv = ld_min_cg(a.t, 1ull << skip);
                for (int j0 = skip; j0 >= 1; j0 -= 8) {
                    double rs[8];
                    float rm[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const int j = j0 - u;
                        rs[u] = j >= 1 ? ld_sum_cg(a.t, (1ull << j) + 1) : 0.0;
                        rm[u] = j >= 1 ? ld_min_cg(a.t, (1ull << j) + 1) : 0.0f;
                    }
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const int j = j0 - u;
                        if (j >= 1) {
                            sv = sv + rs[u];
                            mv = fmin_tree(mv, rm[u]);
                            a.t.S[1ull << (j - 1)] = sv;
                            a.t.M[1ull << (j - 1)] = mv;
                        }
                    }
                }
            }
        }
    }
}

// Subtrees per CTA of the update kernel: one per warp (measured on GB300 against 2 or 1 per
// CTA, which spread the climbs over more SMs: 36.8K and 36.0K against 37.0K apex steps/s).
int update_subtrees_per_cta(int warps) { return warps; }

// Small update grids (at most 16 CTAs) run as one cluster (measured on GB300: the apex step
// 34.3K against 33.9K steps/s with the arrival ticket).
bool update_cluster_enabled() { return true; }

// Target batch entries per subtree of the update kernel: 8 (measured on GB300 against 4 and 2:
// 37.0K against 36.3K and 35.6K apex steps/s).
int update_entries_per_subtree() { return 8; }

int ilog2_ceil(unsigned long long v)
{
    int l = 0;
    while ((1ull << l) < v) ++l;
    return l;
}

}  // namespace

cudaError_t init_tree_kernels(int carveout)
{
    const LeafPowTables tables = make_leaf_pow_tables();
    cudaError_t e = cudaMemcpyToSymbol(g_leafpow, &tables, sizeof(tables));
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(k_update<kUpdWindow>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)update_smem_bytes(kUpdMaxWarps));
    if (e == cudaSuccess) e = cudaFuncSetAttribute(k_update<kUpdWindow>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess || carveout < 0) return e;
    // k_rebuild_tree keeps the driver's choice: its 25 KB of shared memory per CTA would hold it
    // to one CTA per SM in the smallest configuration (a one-entry rebuild of 2^21 leaves took
    // 38.9 us against 22.6 us, of 2^24 leaves 178.7 against 82.5)
    const void *fns[] = {(const void *)k_update<kUpdWindow>, (const void *)k_add, (const void *)k_add_bulk_rows,
                         (const void *)k_add_finish, (const void *)k_fill, (const void *)k_upd_scatter,
                         (const void *)k_upd_apply, (const void *)k_upd_finish, (const void *)k_upd_element};
    for (const void *f : fns) {
        e = cudaFuncSetAttribute(f, cudaFuncAttributePreferredSharedMemoryCarveout, carveout);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t launch_fill_mins(float *M, unsigned long long n, cudaStream_t st)
{
    const unsigned grid = (unsigned)std::min<unsigned long long>((n + kThreads - 1) / kThreads, 4096);
    k_fill<<<grid, kThreads, 0, st>>>(M, n, __builtin_huge_valf());
    return cudaGetLastError();
}

// Both trees rebuilt from the leaves: 11 levels per launch, the last launch's last CTA
// finishing at the root (one launch up to 2^22 leaves, two up to 2^33).  `base` carries the
// large-batch update's winner words and the fold of its maximum (win null for insertions).
cudaError_t launch_rebuild_tree(const RebuildArgs &base, cudaStream_t st)
{
    cudaError_t e = cudaSuccess;
    for (int cd = base.t.D; cd > 0 && e == cudaSuccess; cd -= kRbLog) {
        const unsigned long long grid = cd < kRbLog ? 1 : 1ull << (cd - kRbLog);
        RebuildArgs a = base;
        a.cd = cd;
        if (cd != base.t.D) a.win = nullptr;   // the leaves are done after the first launch
        const bool last = grid <= (unsigned long long)kRbIn;
        a.fold = last ? base.fold : 0;
        e = launch_pdl(k_rebuild_tree, (unsigned)grid, kThreads, 0, st, a);
        if (last) break;
    }
    return e;
}

RebuildArgs rebuild_args(const TreeRefs &t, Ctl *ctl)
{
    RebuildArgs a{};
    a.t = t;
    a.ctl = ctl;
    a.cd = t.D;
    a.win = nullptr;
    a.td = nullptr;
    a.eps = 0.0;
    a.lp = make_leaf_pow_alpha(1.0);
    a.fold = 0;
    a.alpha = 1.0;
    a.crowd = CrowdRefs{nullptr, nullptr, 0, 0};
    return a;
}

cudaError_t launch_add(const TreeRefs &t, const RingRefs &r, float *raw_store, Ctl *ctl,
                       unsigned long long count, const float *states, const float *next,
                       const unsigned *actions, const float *rewards, const unsigned char *dones,
                       const float *prio, double alpha, double eps, bool proportional,
                       unsigned long long host_cursor, int num_sms, const DirtyRefs &dirty,
                       const double *rank_cdf, bool *marked, cudaStream_t st)
{
    (void)host_cursor;
    AddArgs a;
    a.t = t;
    a.r = r;
    a.raw_store = raw_store;
    a.ctl = ctl;
    a.count = count;
    const unsigned long long C = r.capacity;
    a.k0 = count > C ? count - C : 0;
    const unsigned long long cnt = count - a.k0;
    a.states = states;
    a.next = next;
    a.actions = actions;
    a.rewards = rewards;
    a.dones = dones;
    a.prio = prio;
    a.alpha = alpha;
    a.eps = eps;
    a.lp = make_leaf_pow_alpha(alpha);
    a.proportional = proportional ? 1 : 0;
    a.bl = std::min(kAddBlockLog, t.D);
    const unsigned long long bsz = 1ull << a.bl;
    a.vec4 = (r.d % 4 == 0) && ((reinterpret_cast<uintptr_t>(states) | reinterpret_cast<uintptr_t>(next)) % 16 == 0);
    a.rank_cdf = rank_cdf;
    if (r.d == 0) a.vec4 = 0;

    // rows: about `per` elements of each array per copy thread, at most 4 CTAs per SM.  8 (16
    // float4 loads in flight per thread) measured best on GB300 for the apex step: 36.7K steps/s
    // against 35.7K with 2 (128 copy CTAs) and 35.4K with 16.
    constexpr unsigned long long per = 8;
    const unsigned long long elems = a.vec4 ? cnt * (r.d / 4) : cnt * (unsigned long long)std::max(r.d, 1u);
    unsigned ncopy = (unsigned)std::min<unsigned long long>((elems + per * kThreads - 1) / (per * kThreads),
                                                            (unsigned long long)num_sms * 4);
    if (ncopy == 0) ncopy = 1;

    const bool incremental = cnt + bsz <= C && cnt * 8 <= t.n && cnt <= (1ull << 18);
    if (marked) *marked = incremental;
    a.dirty = incremental ? dirty : DirtyRefs{nullptr, nullptr, nullptr, nullptr, nullptr};
    if (incremental) {
        a.ntree = (unsigned)(cnt / bsz + 3);
        a.ncopy = ncopy;
        return launch_pdl(k_add, a.ntree + a.ncopy, kThreads, 0, st, a);
    }
    a.ntree = 0;
    a.ncopy = ncopy;
    cudaError_t e = launch_pdl(k_add_bulk_rows, ncopy, kThreads, 0, st, a);
    if (e != cudaSuccess) return e;
    if (proportional && t.S) {
        e = launch_rebuild_tree(rebuild_args(t, ctl), st);
        if (e != cudaSuccess) return e;
    }
    k_add_finish<<<1, 32, 0, st>>>(ctl, count, C, alpha, rank_cdf);
    return cudaGetLastError();
}

cudaError_t launch_update_element(const TreeRefs &t, Ctl *ctl, unsigned B, const long long *idx,
                                  const float *td, double alpha, double eps, cudaStream_t st)
{
    ElementArgs a;
    a.t = t;
    a.ctl = ctl;
    a.idx = idx;
    a.td = td;
    a.B = B;
    a.alpha = alpha;
    a.eps = eps;
    a.lp = make_leaf_pow_alpha(alpha);
    return launch_pdl(k_upd_element, 1, 32, 0, st, a);
}

cudaError_t launch_update_rebuild(const TreeRefs &t, float *raw_store, Ctl *ctl, unsigned B,
                                  const long long *idx, const float *td, double alpha, double eps,
                                  bool proportional, int num_sms, const DirtyRefs &dirty, unsigned *win,
                                  const CrowdRefs &crowd, cudaStream_t st)
{
    ScatterArgs a;
    a.t = t;
    a.raw_store = raw_store;
    a.ctl = ctl;
    a.dirty = dirty;
    a.win = win;
    a.idx = idx;
    a.td = td;
    a.B = B;
    a.eps = eps;
    a.alpha = alpha;
    a.lp = make_leaf_pow_alpha(alpha);
    a.proportional = proportional ? 1 : 0;
    const bool tree = proportional && t.D > 0 && t.S;
    a.crowd = tree ? crowd : CrowdRefs{nullptr, nullptr, 0, 0};
    if (!tree && B <= kBlockBatch) return launch_pdl_cluster(k_upd_block, kBlockCtas, kBlockThreads, 0, st, a);
    const unsigned grid = (unsigned)std::min<unsigned long long>((B + kThreads - 1) / kThreads,
                                                                 (unsigned long long)num_sms * 8);
    cudaError_t e = launch_pdl(k_upd_scatter, grid, kThreads, 0, st, a);
    if (e != cudaSuccess) return e;
    if (tree) {
        // the leaf level of the rebuild applies the winners and the last CTA folds the maximum
        RebuildArgs r = rebuild_args(t, ctl);
        r.win = win;
        r.td = td;
        r.eps = eps;
        r.lp = a.lp;
        r.fold = 1;
        r.alpha = alpha;
        r.crowd = a.crowd;
        return launch_rebuild_tree(r, st);
    }
    e = launch_pdl(k_upd_apply, grid, kThreads, 0, st, a);
    if (e == cudaSuccess) e = launch_pdl(k_upd_finish, 1, 32, 0, st, ctl, alpha);
    return e;
}

int update_subtree_log(unsigned B, int D)
{
    // about 8 batch entries per subtree (a warp's list holds 512 or 128, so a batch concentrated
    // on a stretch of recent slots still fits; more take the chunked path); at most 2^10
    // subtrees, and no more than half the leaves
    const int per = update_entries_per_subtree();
    int P = ilog2_ceil((B + per - 1) / per);
    P = std::min(P, kMaxTopLog);
    return std::min(P, std::max(D - 1, 0));
}

cudaError_t launch_update(const TreeRefs &t, float *raw_store, Ctl *ctl, unsigned B,
                          const long long *idx, const float *td, double alpha, double eps,
                          bool proportional, int num_sms, const DirtyRefs &dirty, const CrowdRefs &crowd,
                          int P_in, cudaStream_t st)
{
    (void)num_sms;
    UpdArgs a;
    a.t = t;
    a.raw_store = raw_store;
    a.ctl = ctl;
    a.dirty = dirty;
    a.idx = idx;
    a.td = td;
    a.B = B;
    a.pb = std::max(1, ilog2_ceil(B));
    a.alpha = alpha;
    a.eps = eps;
    a.lp = make_leaf_pow_alpha(alpha);
    a.proportional = proportional ? 1 : 0;
    a.crowd_host = proportional && t.S ? crowd.host : nullptr;
    const int P = P_in >= 0 ? std::min(P_in, std::min(kMaxTopLog, std::max(t.D - 1, 0))) : update_subtree_log(B, t.D);
    a.P = P;
    const bool large = B >= kUpdLargeBatch;
    const int warps = large ? kUpdLargeWarps : kUpdSmallWarps;
    a.cap = large ? kUpdLargeCap : kUpdSmallCap;
    a.subs = update_subtrees_per_cta(warps);
    const unsigned grid = (unsigned)(((1ull << P) + a.subs - 1) / a.subs);
    a.cluster = 0;
    if (grid > 1 && grid <= 16 && update_cluster_enabled()) {
        a.cluster = 1;
        return launch_pdl_cluster(k_update<kUpdWindow>, grid, 32 * warps, update_smem_bytes(warps), st, a);
    }
    return launch_pdl(k_update<kUpdWindow>, grid, 32 * warps, update_smem_bytes(warps), st, a);
}

}  // namespace gbper
