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

#include <algorithm>

namespace gbper {

namespace {

constexpr int kThreads = 256;
constexpr int kAddBlockLog = 8;      // leaves per tree CTA in the insertion kernel: 256
constexpr int kTopSpan = 1040;       // widest dirty span the last CTA handles on insertion
constexpr int kUpdCap = 1024;        // batch entries one update CTA sorts in shared memory
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

// Arrival ticket: returns true in every thread of the last CTA to arrive.  No CTA waits.
__device__ __forceinline__ bool last_to_arrive(unsigned *ticket)
{
    __shared__ int s_last;
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        const unsigned t = atomicAdd(ticket, 1u);
        s_last = (t == gridDim.x - 1);
    }
    __syncthreads();
    const bool last = s_last;
    if (last) __threadfence();
    return last;
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
__device__ void top_range_upsweep(const TreeRefs &t, int L0, unsigned long long lo,
                                  unsigned long long hi, double *spS0, float *spM0,
                                  double *spS1, float *spM1, double *exS, float *exM)
{
    if (L0 <= 0) return;
    const unsigned long long lvl0 = 1ull << L0;
    // span at depth L0: [2(lo>>1), 2(hi>>1)+1]
    unsigned long long sp_lo = (lo >> 1) << 1;
    unsigned long long sp_hi = ((hi >> 1) << 1) + 1;
    const int w0 = (int)(sp_hi - sp_lo + 1);
    for (int i = threadIdx.x; i < w0; i += blockDim.x) {
        spS0[i] = ld_sum_cg(t, lvl0 + sp_lo + i);
        spM0[i] = ld_min_cg(t, lvl0 + sp_lo + i);
    }
    // clean edge siblings of depths L0-1 .. 1: slot 2l (left) and 2l+1 (right)
    for (int l = 1 + (int)threadIdx.x; l < L0; l += blockDim.x) {
        const unsigned long long a = lo >> (L0 - l), b = hi >> (L0 - l);
        const unsigned long long base = 1ull << l;
        if (a & 1ull) { exS[2 * l] = ld_sum_cg(t, base + a - 1); exM[2 * l] = ld_min_cg(t, base + a - 1); }
        if (!(b & 1ull)) { exS[2 * l + 1] = ld_sum_cg(t, base + b + 1); exM[2 * l + 1] = ld_min_cg(t, base + b + 1); }
    }
    __syncthreads();
    double *curS = spS0, *nxtS = spS1;
    float *curM = spM0, *nxtM = spM1;
    unsigned long long a = lo, b = hi;  // dirty range at the current depth
    for (int l = L0; l >= 1; --l) {
        const unsigned long long pa = a >> 1, pb = b >> 1;      // dirty parents at depth l-1
        const int np = (int)(pb - pa + 1);
        // next span at depth l-1 (only needed when l-1 >= 1)
        const unsigned long long nsp_lo = (pa >> 1) << 1;
        const unsigned long long pbase = 1ull << (l - 1);
        for (int i = threadIdx.x; i < np; i += blockDim.x) {
            const unsigned long long p = pa + i;
            const int c = (int)(2 * p - sp_lo);
            const double s = curS[c] + curS[c + 1];
            const float m = fmin_tree(curM[c], curM[c + 1]);
            t.S[pbase + p] = s;
            t.M[pbase + p] = m;
            nxtS[p - nsp_lo] = s;
            nxtM[p - nsp_lo] = m;
        }
        if (threadIdx.x == 0 && l - 1 >= 1) {
            if (pa & 1ull) { nxtS[0] = exS[2 * (l - 1)]; nxtM[0] = exM[2 * (l - 1)]; }
            if (!(pb & 1ull)) {
                const int r = (int)(pb + 1 - nsp_lo);
                nxtS[r] = exS[2 * (l - 1) + 1];
                nxtM[r] = exM[2 * (l - 1) + 1];
            }
        }
        __syncthreads();
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
    unsigned long long count, k0;
    const float *states, *next;
    const unsigned *actions;
    const float *rewards;
    const unsigned char *dones;
    const float *prio;
    double alpha, eps;
    int proportional;
    int bl;            // log2 leaves per tree block
    unsigned ntree;    // tree CTAs (upper bound over cursor positions)
    unsigned ncopy;    // row-copy CTAs
    int vec4;          // rows copy as float4
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

__global__ void __launch_bounds__(kThreads) k_add(AddArgs a)
{
    __shared__ double s_vs[1 << kAddBlockLog];
    __shared__ float s_vm[1 << kAddBlockLog];
    const unsigned long long cursor = a.ctl->cursor;
    const float max_prev = __uint_as_float(a.ctl->max_raw_bits);
    const unsigned long long C = a.r.capacity;
    const AddGeom g = add_geometry(a, cursor);
    const int tid = threadIdx.x;

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
                        leaf = raw_to_leaf(raw, a.alpha);
                        a.t.L[s] = leaf;
                    } else {
                        a.raw_store[s] = raw;
                    }
                } else if (a.proportional) {
                    leaf = a.t.L[s];
                }
                if (a.proportional) {
                    s_vs[tid] = (double)leaf;
                    s_vm[tid] = leaf_min_value(leaf);
                }
            }
            if (a.proportional) {
                const unsigned long long first = a.t.n + ((unsigned long long)blk << a.bl);
                for (int h = 1; h <= a.bl; ++h) {
                    const int cnt = bsz >> h;
                    double sv = 0.0;
                    float mv = 0.0f;
                    __syncthreads();
                    if (tid < cnt) {
                        sv = s_vs[2 * tid] + s_vs[2 * tid + 1];
                        mv = fmin_tree(s_vm[2 * tid], s_vm[2 * tid + 1]);
                    }
                    __syncthreads();
                    if (tid < cnt) {
                        s_vs[tid] = sv;
                        s_vm[tid] = mv;
                        const unsigned long long node = (first >> h) + tid;
                        a.t.S[node] = sv;
                        a.t.M[node] = mv;
                    }
                }
            }
        }
        const unsigned bm = block_max_u32(mymax);
        if (tid == 0 && bm) atomicMax(&a.ctl->add_max_bits, bm);
    } else {
        // rows that a later row of the same call overwrites still count toward the running
        // maximum, as if they had been inserted one after another
        unsigned mymax = 0;
        if (a.prio) {
            const unsigned long long t0 = (unsigned long long)(blockIdx.x - a.ntree) * kThreads + tid;
            for (unsigned long long k = t0; k < a.k0; k += (unsigned long long)a.ncopy * kThreads)
                mymax = max(mymax, __float_as_uint(prio_to_raw(__ldg(a.prio + k), a.eps, max_prev)));
        }
        const unsigned bm = block_max_u32(mymax);
        if (tid == 0 && bm) atomicMax(&a.ctl->add_max_bits, bm);
        // row copies: one warp per row, rows strided over the copy CTAs
        const unsigned long long cnt = a.count - a.k0;
        const int warp = tid >> 5, lane = tid & 31;
        const unsigned long long wglob = (unsigned long long)(blockIdx.x - a.ntree) * (kThreads / 32) + warp;
        const unsigned long long wtotal = (unsigned long long)a.ncopy * (kThreads / 32);
        for (unsigned long long o = wglob; o < cnt; o += wtotal) {
            const unsigned long long k = a.k0 + o;
            const unsigned long long slot = (g.s0 + o) % C;
            if (a.r.d) copy_row(a, k, slot, lane, 32);
            if (lane == 0) {
                a.r.actions[slot] = __ldg(a.actions + k);
                a.r.rewards[slot] = __ldg(a.rewards + k);
                a.r.dones[slot] = __ldg(a.dones + k);
            }
        }
    }

    if (last_to_arrive(&a.ctl->ticket_add)) {
        if (a.proportional) {
            __shared__ double s_spS0[kTopSpan], s_spS1[kTopSpan];
            __shared__ float s_spM0[kTopSpan], s_spM1[kTopSpan];
            __shared__ double s_exS[64];
            __shared__ float s_exM[64];
            const int L0 = a.t.D - a.bl;
            top_range_upsweep(a.t, L0, g.blkA0, g.blkA0 + g.nA - 1, s_spS0, s_spM0, s_spS1,
                              s_spM1, s_exS, s_exM);
            if (g.nB) {
                __syncthreads();
                top_range_upsweep(a.t, L0, 0, g.nB - 1, s_spS0, s_spM0, s_spS1, s_spM1, s_exS,
                                  s_exM);
            }
        }
        if (tid == 0) {
            Ctl *c = a.ctl;
            const unsigned am = __ldcg(&c->add_max_bits);
            if (am > c->max_raw_bits) c->max_raw_bits = am;
            c->add_max_bits = 0;
            c->cursor = (cursor + a.count) % C;
            const unsigned long long sz = c->size + a.count;
            c->size = sz < C ? sz : C;
            c->ticket_add = 0;
        }
    }
}

// ---- bulk insertion: rows + leaves, then a full level-by-level rebuild -------------------

__global__ void __launch_bounds__(kThreads) k_add_bulk_rows(AddArgs a)
{
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
            if (a.proportional) a.t.L[slot] = raw_to_leaf(raw, a.alpha);
            else a.raw_store[slot] = raw;
        }
    }
    const unsigned bm = block_max_u32(mymax);
    if (threadIdx.x == 0 && bm) atomicMax(&a.ctl->add_max_bits, bm);
}

// Rebuild every node from depth cd-1 up to depth pd (pd < cd) from the nodes at depth cd.
// Each CTA owns 256 consecutive nodes at depth cd (or the whole level when it is smaller).
__global__ void __launch_bounds__(kThreads) k_rebuild_levels(TreeRefs t, int cd, int pd)
{
    __shared__ double s_vs[kThreads];
    __shared__ float s_vm[kThreads];
    const unsigned long long width = 1ull << cd;
    const int gl = cd - pd;  // levels this launch builds (<= 8)
    const unsigned long long first = width + (unsigned long long)blockIdx.x * kThreads;
    const int tid = threadIdx.x;
    const int bsz = width < (unsigned long long)kThreads ? (int)width : kThreads;
    if (tid < bsz) {
        s_vs[tid] = ld_sum(t, first + tid);
        s_vm[tid] = ld_min(t, first + tid);
    }
    for (int h = 1; h <= gl; ++h) {
        const int cnt = bsz >> h;
        double sv = 0.0;
        float mv = 0.0f;
        __syncthreads();
        if (tid < cnt) {
            sv = s_vs[2 * tid] + s_vs[2 * tid + 1];
            mv = fmin_tree(s_vm[2 * tid], s_vm[2 * tid + 1]);
        }
        __syncthreads();
        if (tid < cnt) {
            s_vs[tid] = sv;
            s_vm[tid] = mv;
            const unsigned long long node = (first >> h) + tid;
            t.S[node] = sv;
            t.M[node] = mv;
        }
    }
}

__global__ void k_add_finish(Ctl *c, unsigned long long count, unsigned long long C)
{
    if (threadIdx.x == 0 && blockIdx.x == 0) {
        const unsigned am = c->add_max_bits;
        if (am > c->max_raw_bits) c->max_raw_bits = am;
        c->add_max_bits = 0;
        c->cursor = (c->cursor + count) % C;
        const unsigned long long sz = c->size + count;
        c->size = sz < C ? sz : C;
    }
}

__global__ void k_fill(float *p, unsigned long long n, float v)
{
    for (unsigned long long i = blockIdx.x * (unsigned long long)blockDim.x + threadIdx.x; i < n;
         i += (unsigned long long)gridDim.x * blockDim.x)
        p[i] = v;
}

// ------------------------------------------------------------------------------------------
// Priority update: last-writer-wins scatter + dirty-ancestor upsweep, one launch.
// CTA c owns the subtree at depth P whose leaves are [c << shift, (c+1) << shift).  It reads
// the whole batch, keeps the entries in its subtree, sorts them by (leaf, batch position) in
// shared memory, keeps the last position of each leaf, writes those leaves, and climbs its
// subtree level by level.  On each level the first entry of every run of entries below the
// same node owns that node; the owner of a left child reaches the owner of a dirty right
// sibling through a run-end pointer (pointer jumping), and clean siblings come from global
// memory, loaded for a window of levels before the window is combined.  The last CTA to
// arrive rebuilds the 2^P - 1 nodes above the subtree roots and folds the batch maximum into
// the running maximum.
// ------------------------------------------------------------------------------------------
struct UpdArgs {
    TreeRefs t;
    float *raw_store;
    Ctl *ctl;
    const long long *idx;
    const float *td;
    unsigned B;
    int P;      // log2 grid size
    int pb;     // bits for a batch position
    double alpha, eps;
    int proportional;
};

struct UpdSmem {
    unsigned long long *keys;  // [cap] (leaf offset << pb) | position
    unsigned *pay;             // [cap] entry slot carried through the sort
    float *rawv;               // [cap] raw priority by entry slot
    unsigned *ulist;           // [cap] sorted distinct leaves (absolute)
    float *uleaf;              // [cap] new leaf value (sum/min seed)
    double *vs;                // [cap]
    float *vm;                 // [cap]
    int *rend;                 // [cap]
    int *flag;                 // [cap + 1] winner flags -> exclusive scan
    double *heapS;             // [2^(kMaxTopLog+1)]
    float *heapM;
};

__device__ __forceinline__ UpdSmem upd_smem_layout(unsigned char *base)
{
    UpdSmem s;
    s.keys = reinterpret_cast<unsigned long long *>(base);
    s.vs = reinterpret_cast<double *>(s.keys + kUpdCap);
    s.heapS = s.vs + kUpdCap;
    unsigned char *p = reinterpret_cast<unsigned char *>(s.heapS + (2 << kMaxTopLog));
    s.pay = reinterpret_cast<unsigned *>(p);
    s.rawv = reinterpret_cast<float *>(s.pay + kUpdCap);
    s.ulist = reinterpret_cast<unsigned *>(s.rawv + kUpdCap);
    s.uleaf = reinterpret_cast<float *>(s.ulist + kUpdCap);
    s.vm = s.uleaf + kUpdCap;
    s.rend = reinterpret_cast<int *>(s.vm + kUpdCap);
    s.flag = s.rend + kUpdCap;
    s.heapM = reinterpret_cast<float *>(s.flag + kUpdCap + 32);
    return s;
}

constexpr size_t kUpdSmemBytes =
    (size_t)kUpdCap * 8 * 2 + (size_t)(2 << kMaxTopLog) * 8 +
    (size_t)kUpdCap * 4 * 7 + 32 * 4 + (size_t)(2 << kMaxTopLog) * 4;

// Bitonic sort of keys[0, m2) (m2 a power of two) carrying pay[]; ascending.
__device__ void bitonic_sort_kv(unsigned long long *keys, unsigned *pay, int m2)
{
    for (int k = 2; k <= m2; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int t = threadIdx.x; t < (m2 >> 1); t += blockDim.x) {
                const int i = (t / j) * 2 * j + (t % j);
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
            __syncthreads();
        }
    }
}

// Exclusive scan of flag[0, m) in place; returns the total (valid in all threads).
__device__ int block_exclusive_scan(int *flag, int m)
{
    __shared__ int s_warp[kThreads / 32];
    __shared__ int s_total;
    const int per = (m + blockDim.x - 1) / blockDim.x;
    const int beg = threadIdx.x * per;
    int sum = 0;
    for (int i = 0; i < per; ++i)
        if (beg + i < m) sum += flag[beg + i];
    // warp inclusive scan of per-thread sums
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = sum;
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    if (threadIdx.x == 0) {
        int run = 0;
        for (int w = 0; w < (int)(blockDim.x >> 5); ++w) {
            const int v = s_warp[w];
            s_warp[w] = run;
            run += v;
        }
        s_total = run;
    }
    __syncthreads();
    int run = s_warp[warp] + incl - sum;
    for (int i = 0; i < per; ++i)
        if (beg + i < m) {
            const int v = flag[beg + i];
            flag[beg + i] = run;
            run += v;
        }
    __syncthreads();
    return s_total;
}

template <int W>
__global__ void __launch_bounds__(kThreads) k_update(UpdArgs a)
{
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const UpdSmem sm = upd_smem_layout(smem_raw);
    __shared__ int s_count;
    __shared__ unsigned s_max;
    const int tid = threadIdx.x;
    const int D = a.t.D;
    const int shift = D - a.P;
    const unsigned long long c = blockIdx.x;
    const unsigned long long base = c << shift;
    const unsigned long long n = a.t.n;
    const unsigned long long size = a.ctl->size;
    const float max_prev = __uint_as_float(a.ctl->max_raw_bits);
    if (tid == 0) {
        s_count = 0;
        s_max = 0;
    }
    __syncthreads();

    // 1. keep this subtree's entries
    for (unsigned j = tid; j < a.B; j += blockDim.x) {
        const long long i = __ldg(a.idx + j);
        if (i < 0 || (unsigned long long)i >= size) {
            if (c == 0) atomicOr(&a.ctl->err_flags, kFlagBadIndex);
            continue;
        }
        if (((unsigned long long)i >> shift) != c) continue;
        const float raw = td_to_raw(__ldg(a.td + j), a.eps, max_prev);
        atomicMax(&s_max, __float_as_uint(raw));
        const int slot = atomicAdd(&s_count, 1);
        if (slot < kUpdCap) {
            sm.keys[slot] = (((unsigned long long)i - base) << a.pb) | j;
            sm.pay[slot] = (unsigned)slot;
            sm.rawv[slot] = raw;
        }
    }
    __syncthreads();
    const int m = s_count;
    if (tid == 0 && s_max) atomicMax(&a.ctl->batch_max_bits, s_max);

    if (m > kUpdCap) {
        // Rare: more entries than one CTA sorts at once.  Apply the batch in position order,
        // chunk by chunk (a later chunk overwrites an earlier one: last writer wins), then
        // rebuild this whole subtree level by level.
        for (unsigned p0 = 0; p0 < a.B; p0 += blockDim.x) {
            if (tid == 0) s_count = 0;
            __syncthreads();
            const unsigned j = p0 + tid;
            if (j < a.B) {
                const long long i = __ldg(a.idx + j);
                if (i >= 0 && (unsigned long long)i < size && ((unsigned long long)i >> shift) == c) {
                    const int slot = atomicAdd(&s_count, 1);
                    sm.keys[slot] = (((unsigned long long)i - base) << a.pb) | j;
                    sm.pay[slot] = (unsigned)slot;
                    sm.rawv[slot] = td_to_raw(__ldg(a.td + j), a.eps, max_prev);
                }
            }
            __syncthreads();
            const int mc = s_count;
            if (mc > 0) {
                int m2 = 1;
                while (m2 < mc) m2 <<= 1;
                for (int i = mc + tid; i < m2; i += blockDim.x) sm.keys[i] = ~0ull;
                __syncthreads();
                bitonic_sort_kv(sm.keys, sm.pay, m2);
                for (int k = tid; k < mc; k += blockDim.x) {
                    const unsigned long long lk = sm.keys[k] >> a.pb;
                    if (k == mc - 1 || (sm.keys[k + 1] >> a.pb) != lk) {
                        const unsigned long long leaf = base + lk;
                        const float raw = sm.rawv[sm.pay[k]];
                        if (a.proportional) a.t.L[leaf] = raw_to_leaf(raw, a.alpha);
                        else a.raw_store[leaf] = raw;
                    }
                }
            }
            __syncthreads();
        }
        if (a.proportional) {
            for (int h = 1; h <= shift; ++h) {
                const unsigned long long cnt = 1ull << (shift - h);
                const unsigned long long first = (n + base) >> h;
                for (unsigned long long q = tid; q < cnt; q += blockDim.x) {
                    const unsigned long long node = first + q;
                    a.t.S[node] = ld_sum(a.t, 2 * node) + ld_sum(a.t, 2 * node + 1);
                    a.t.M[node] = fmin_tree(ld_min(a.t, 2 * node), ld_min(a.t, 2 * node + 1));
                }
                __syncthreads();
            }
        }
    } else if (m > 0) {
        int m2 = 2;
        while (m2 < m) m2 <<= 1;
        for (int i = m + tid; i < m2; i += blockDim.x) sm.keys[i] = ~0ull;
        __syncthreads();
        bitonic_sort_kv(sm.keys, sm.pay, m2);
        // 2. winners: the last position of each leaf
        for (int k = tid; k < m; k += blockDim.x)
            sm.flag[k] = (k == m - 1 || (sm.keys[k + 1] >> a.pb) != (sm.keys[k] >> a.pb)) ? 1 : 0;
        __syncthreads();
        const int U = block_exclusive_scan(sm.flag, m);
        for (int k = tid; k < m; k += blockDim.x) {
            const bool win = (k == m - 1) || (sm.flag[k + 1] != sm.flag[k]);
            if (win) {
                const int u = sm.flag[k];
                const unsigned long long leaf = base + (sm.keys[k] >> a.pb);
                const float raw = sm.rawv[sm.pay[k]];
                sm.ulist[u] = (unsigned)leaf;
                if (a.proportional) {
                    const float lv = raw_to_leaf(raw, a.alpha);
                    a.t.L[leaf] = lv;
                    sm.vs[u] = (double)lv;
                    sm.vm[u] = leaf_min_value(lv);
                    sm.rend[u] = u + 1;
                } else {
                    a.raw_store[leaf] = raw;
                }
            }
        }
        __syncthreads();

        // 3. climb from the leaves (h = 0) to the subtree root at depth P
        if (a.proportional) {
            const int R = (U + blockDim.x - 1) / blockDim.x;
            if (R == 1) {
                // one entry per thread: clean siblings of W levels are loaded up front
                const int k = tid;
                const bool have = k < U;
                const unsigned long long myleaf = have ? (unsigned long long)sm.ulist[k] + n : 0;
                const unsigned long long prevleaf = (have && k > 0) ? (unsigned long long)sm.ulist[k - 1] + n : 0;
                for (int h0 = 0; h0 < shift; h0 += W) {
                    double ps[W];
                    float pmn[W];
#pragma unroll
                    for (int w = 0; w < W; ++w) {
                        const int h = h0 + w;
                        ps[w] = 0.0;
                        pmn[w] = 0.0f;
                        if (have && h < shift) {
                            const unsigned long long v = myleaf >> h;
                            const bool owner = (k == 0) || ((prevleaf >> h) != v);
                            if (owner) {
                                ps[w] = ld_sum(a.t, v ^ 1ull);
                                pmn[w] = ld_min(a.t, v ^ 1ull);
                            }
                        }
                    }
#pragma unroll
                    for (int w = 0; w < W; ++w) {
                        const int h = h0 + w;
                        if (h < shift) {
                            if (have) {
                                const unsigned long long v = myleaf >> h;
                                const bool owner = (k == 0) || ((prevleaf >> h) != v);
                                if (owner) {
                                    const double ms = sm.vs[k];
                                    const float mm = sm.vm[k];
                                    bool compute = true;
                                    double s;
                                    float mn;
                                    int ne = sm.rend[k];
                                    if ((v & 1ull) == 0) {
                                        const int e = ne;
                                        if (e < U && ((((unsigned long long)sm.ulist[e] + n) >> h) == v + 1)) {
                                            s = ms + sm.vs[e];
                                            mn = fmin_tree(mm, sm.vm[e]);
                                            ne = sm.rend[e];
                                        } else {
                                            s = ms + ps[w];
                                            mn = fmin_tree(mm, pmn[w]);
                                        }
                                    } else {
                                        if (k > 0 && ((prevleaf >> h) == v - 1)) {
                                            compute = false;
                                        } else {
                                            s = ps[w] + ms;
                                            mn = fmin_tree(pmn[w], mm);
                                        }
                                    }
                                    if (compute) {
                                        sm.vs[k] = s;
                                        sm.vm[k] = mn;
                                        sm.rend[k] = ne;
                                        a.t.S[v >> 1] = s;
                                        a.t.M[v >> 1] = mn;
                                    }
                                }
                            }
                            __syncthreads();
                        }
                    }
                }
            } else {
                for (int h = 0; h < shift; ++h) {
                    for (int k = tid; k < U; k += blockDim.x) {
                        const unsigned long long v = ((unsigned long long)sm.ulist[k] + n) >> h;
                        const bool owner = (k == 0) || (((((unsigned long long)sm.ulist[k - 1]) + n) >> h) != v);
                        if (!owner) continue;
                        const double ms = sm.vs[k];
                        const float mm = sm.vm[k];
                        int ne = sm.rend[k];
                        double s;
                        float mn;
                        if ((v & 1ull) == 0) {
                            const int e = ne;
                            if (e < U && ((((unsigned long long)sm.ulist[e] + n) >> h) == v + 1)) {
                                s = ms + sm.vs[e];
                                mn = fmin_tree(mm, sm.vm[e]);
                                ne = sm.rend[e];
                            } else {
                                s = ms + ld_sum(a.t, v + 1);
                                mn = fmin_tree(mm, ld_min(a.t, v + 1));
                            }
                        } else {
                            if (k > 0 && ((((unsigned long long)sm.ulist[k - 1] + n) >> h) == v - 1)) continue;
                            s = ld_sum(a.t, v - 1) + ms;
                            mn = fmin_tree(ld_min(a.t, v - 1), mm);
                        }
                        sm.vs[k] = s;
                        sm.vm[k] = mn;
                        sm.rend[k] = ne;
                        a.t.S[v >> 1] = s;
                        a.t.M[v >> 1] = mn;
                    }
                    __syncthreads();
                }
            }
        }
    }

    // 4. the last CTA rebuilds the top P levels and folds in the batch maximum
    if (last_to_arrive(&a.ctl->ticket_update)) {
        if (a.proportional && a.P > 0) {
            const int P = a.P;
            const int width = 1 << P;
            for (int i = tid; i < width; i += blockDim.x) {
                sm.heapS[width + i] = ld_sum_cg(a.t, (unsigned long long)width + i);
                sm.heapM[width + i] = ld_min_cg(a.t, (unsigned long long)width + i);
            }
            for (int l = P - 1; l >= 0; --l) {
                __syncthreads();
                const int lw = 1 << l;
                for (int i = tid; i < lw; i += blockDim.x) {
                    const int node = lw + i;
                    const double s = sm.heapS[2 * node] + sm.heapS[2 * node + 1];
                    const float mn = fmin_tree(sm.heapM[2 * node], sm.heapM[2 * node + 1]);
                    sm.heapS[node] = s;
                    sm.heapM[node] = mn;
                    a.t.S[node] = s;
                    a.t.M[node] = mn;
                }
            }
        }
        if (tid == 0) {
            Ctl *cc = a.ctl;
            const unsigned bm = __ldcg(&cc->batch_max_bits);
            if (bm > cc->max_raw_bits) cc->max_raw_bits = bm;
            cc->batch_max_bits = 0;
            cc->ticket_update = 0;
        }
    }
}

int ilog2_ceil(unsigned long long v)
{
    int l = 0;
    while ((1ull << l) < v) ++l;
    return l;
}

}  // namespace

cudaError_t launch_fill_mins(float *M, unsigned long long n, cudaStream_t st)
{
    const unsigned grid = (unsigned)std::min<unsigned long long>((n + kThreads - 1) / kThreads, 4096);
    k_fill<<<grid, kThreads, 0, st>>>(M, n, __builtin_huge_valf());
    return cudaGetLastError();
}

cudaError_t launch_add(const TreeRefs &t, const RingRefs &r, float *raw_store, Ctl *ctl,
                       unsigned long long count, const float *states, const float *next,
                       const unsigned *actions, const float *rewards, const unsigned char *dones,
                       const float *prio, double alpha, double eps, bool proportional,
                       unsigned long long host_cursor, int num_sms, cudaStream_t st)
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
    a.proportional = proportional ? 1 : 0;
    a.bl = std::min(kAddBlockLog, t.D);
    const unsigned long long bsz = 1ull << a.bl;
    a.vec4 = (r.d % 4 == 0) && ((reinterpret_cast<uintptr_t>(states) | reinterpret_cast<uintptr_t>(next)) % 16 == 0);
    if (r.d == 0) a.vec4 = 0;

    // rows: aim for ~8 rows per warp, at most 4 CTAs per SM
    const unsigned long long warps = (cnt + 7) / 8;
    unsigned ncopy = (unsigned)std::min<unsigned long long>((warps + 7) / 8, (unsigned long long)num_sms * 4);
    if (ncopy == 0) ncopy = 1;

    const bool incremental = cnt + bsz <= C && cnt * 8 <= t.n && cnt <= (1ull << 18);
    if (incremental) {
        a.ntree = (unsigned)(cnt / bsz + 3);
        a.ncopy = ncopy;
        k_add<<<a.ntree + a.ncopy, kThreads, 0, st>>>(a);
        return cudaGetLastError();
    }
    a.ntree = 0;
    a.ncopy = ncopy;
    k_add_bulk_rows<<<ncopy, kThreads, 0, st>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (proportional) {
        for (int cd = t.D; cd > 0; cd -= 8) {
            const int pd = std::max(cd - 8, 0);
            const unsigned long long width = 1ull << cd;
            const unsigned grid = (unsigned)((width + kThreads - 1) / kThreads);
            k_rebuild_levels<<<grid, kThreads, 0, st>>>(t, cd, pd);
            e = cudaGetLastError();
            if (e != cudaSuccess) return e;
        }
    }
    k_add_finish<<<1, 32, 0, st>>>(ctl, count, C);
    return cudaGetLastError();
}

cudaError_t launch_update(const TreeRefs &t, float *raw_store, Ctl *ctl, unsigned B,
                          const long long *idx, const float *td, double alpha, double eps,
                          bool proportional, int num_sms, cudaStream_t st)
{
    (void)num_sms;
    UpdArgs a;
    a.t = t;
    a.raw_store = raw_store;
    a.ctl = ctl;
    a.idx = idx;
    a.td = td;
    a.B = B;
    a.pb = std::max(1, ilog2_ceil(B));
    a.alpha = alpha;
    a.eps = eps;
    a.proportional = proportional ? 1 : 0;
    // ~32 batch entries per CTA; the grid never exceeds 2^10 CTAs or half the leaves
    int P = ilog2_ceil((B + 31) / 32);
    P = std::min(P, kMaxTopLog);
    P = std::min(P, std::max(t.D - 1, 0));
    a.P = P;
    static bool attr_set = false;
    if (!attr_set) {
        cudaFuncSetAttribute(k_update<8>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kUpdSmemBytes);
        attr_set = true;
    }
    k_update<8><<<1u << P, kThreads, kUpdSmemBytes, st>>>(a);
    return cudaGetLastError();
}

}  // namespace gbper
