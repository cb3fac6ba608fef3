/*
 * per_oracle.c -- the oracle for GPU-resident prioritized experience replay (PER).
 *
 * TEST INFRASTRUCTURE ONLY.  A plain, slow, sequential CPU implementation that the tests,
 * the smoke check and the benchmark's CPU-baseline leg load through ctypes.  The CUDA library
 * never links, includes or calls it, and it shares nothing with the CUDA library.
 *
 * Sources, cited by page title and section:
 *   [SEG] "Putting prioritized replay's segment tree on a GPU":
 *         "The Tree Under Every Prioritized Replay" (sum tree in a flat array of length 2n,
 *         internal node = sum of its children, root = total; twin min tree),
 *         "Sampling Is a Descent" (the st_find_prefixsum_idx walk),
 *         "Second Port: Make the Update GPU-Shaped" (leaf writes, then level rebuild), and the
 *         per-element leaf-to-root propagation it compares against.
 *   [GPR] "GPU-Resident Prioritized Experience Replay" (foxhunt design):
 *         "Architecture" (fixed-capacity ring of states, next_states, actions, rewards, dones),
 *         "Sampling Kernels" / Proportional steps 1-5 (uniforms, gather, IS weight
 *         w_i = (1/(N * p_i/total))^beta / max_weight) and Rank-based steps 1-2,
 *         "Priority update" (scatter of the transformed TD error),
 *         "Experience Insertion" (new rows get the maximum priority, cursor wraps),
 *         "Error Handling & Fallback" (NaN/Inf priorities clamped to [epsilon, max_priority]).
 *   [PHX] Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3", SC'11:
 *         the Philox4x32 bijection with ten rounds.
 *
 * Readings taken where the pages leave a step open (each is also listed in the design notes):
 *   R1 internal sums are binary64, leaves binary32 p^alpha; S[i] = S[2i] + S[2i+1] exactly.
 *   R2 raw priority from a TD error: fl32(|td| + eps); leaf = fl32(pow(raw, alpha)) in binary64.
 *   R3 NaN -> eps; +Inf -> the running maximum raw priority as it stood when the call began;
 *      finite values below eps are raised to eps; finite values are never capped.
 *   R4 the running maximum starts at 1.0 and takes every raw priority written (all batch
 *      positions, duplicates included).
 *   R5 draws are stratified: mass_j = (j + u_j) * (T / B).
 *   R6 a mass equal to the left sum goes right (the descent's strict ">"), so the chosen leaf i
 *      satisfies C(i-1) <= mass < C(i).
 *   R7 a descent that lands past the filled slots (rounding at the top end) is clamped to the
 *      last filled slot; the draw counts as near a boundary.
 *   R8 IS weight w = (n P(i))^-beta / max_w with max_w from the min tree reduces to
 *      w = (L[i] / p_min)^-beta; n cancels.
 *   R9 duplicate indices in one update: the highest batch position wins (sequential order).
 *   R10 capacity is rounded up to a power of two; padding leaves hold 0 (sum) and count as
 *      +inf in the min tree.  A leaf of 0 marks an empty slot.
 *   R11 rank mode: rank 1 is the largest raw priority, ties by ascending index;
 *      P(r) = r^-alpha / sum_{k<=size} k^-alpha; w = (r / size)^(alpha * beta).
 *   R12 an update index outside [0, size) is skipped and counted.
 *   R24 uniform mode (the plain replay the pages' PER replaces): every filled slot weighs 1, so
 *      the stratified draw j (stream tag 2) takes mass (j + u_j) * (size / B) and slot
 *      floor(mass), weight 1; insertion stores rows (and follows the running maximum as in the
 *      other modes); updates change nothing.
 *   R26 flat mode (the foxhunt design's own proportional sampler, [GPR] "Sampling Kernels",
 *      Proportional steps 2-3): the same leaves and the same stratified draws as proportional
 *      mode (stream tag 0), but no tree: at each sample the cumulative array
 *      C[i] = C[i-1] + L[i] is summed left to right in binary64 over the filled slots, and draw
 *      j takes the first i with C[i] > mass_j (binary search).  T = C[size-1]; p_min is the
 *      smallest filled leaf; weights as R8.  Updates write leaves only.
 */
#include "per_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

struct orc_per {
    uint64_t capacity; /* ring slots */
    uint64_t n;        /* tree leaves, power of two >= capacity */
    uint32_t d, dp;
    double alpha, eps;
    uint32_t mode;
    uint64_t seed;
    int with_ring;
    /* proportional mode: binary32 leaves, binary64 sums, binary32 mins (index 1..n-1) */
    float *L;
    double *S;
    float *M;
    /* rank mode: raw priorities and the rank CDF */
    float *raw;
    double *cdf;
    /* ring mirror */
    float *states, *next;
    uint32_t *actions;
    float *rewards;
    uint8_t *dones;
    uint64_t size, cursor, calls;
    float max_raw;
};

/* ------------------------------------------------------------------------------------------
 * Philox4x32-10 [PHX].  One round maps (c0,c1,c2,c3) with key (k0,k1) to
 *   (hi(M1*c2) ^ c1 ^ k0,  lo(M1*c2),  hi(M0*c0) ^ c3 ^ k1,  lo(M0*c0)),
 * and the key advances by the Weyl constants between rounds.
 * ------------------------------------------------------------------------------------------ */
void orc_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4])
{
    const uint32_t mult0 = 0xD2511F53u, mult1 = 0xCD9E8D57u;
    const uint32_t weyl0 = 0x9E3779B9u, weyl1 = 0xBB67AE85u;
    uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
    uint32_t k0 = key[0], k1 = key[1];
    for (int round = 0; round < 10; ++round) {
        uint64_t prod0 = (uint64_t)mult0 * (uint64_t)c0;
        uint64_t prod1 = (uint64_t)mult1 * (uint64_t)c2;
        uint32_t hi0 = (uint32_t)(prod0 >> 32), lo0 = (uint32_t)prod0;
        uint32_t hi1 = (uint32_t)(prod1 >> 32), lo1 = (uint32_t)prod1;
        uint32_t n0 = hi1 ^ c1 ^ k0;
        uint32_t n1 = lo1;
        uint32_t n2 = hi0 ^ c3 ^ k1;
        uint32_t n3 = lo0;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
        k0 += weyl0;
        k1 += weyl1;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

double orc_uniform53(uint64_t seed, uint32_t j, uint64_t call, uint32_t tag)
{
    uint32_t ctr[4] = {j, (uint32_t)call, (uint32_t)(call >> 32), tag};
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t x[4];
    orc_philox4x32_10(ctr, key, x);
    uint64_t bits = ((uint64_t)x[0] << 21) | ((uint64_t)x[1] >> 11);
    return (double)bits * 0x1.0p-53;
}

/* ------------------------------------------------------------------------------------------
 * Tree [SEG "The Tree Under Every Prioritized Replay"].  Node 1 is the root, node i has
 * children 2i and 2i+1, and nodes n..2n-1 are the leaves L[0..n-1].
 * ------------------------------------------------------------------------------------------ */
static double node_sum(const orc_per *o, uint64_t i)
{
    return i >= o->n ? (double)o->L[i - o->n] : o->S[i];
}

static float node_min(const orc_per *o, uint64_t i)
{
    if (i >= o->n) {
        float v = o->L[i - o->n];
        return v > 0.0f ? v : INFINITY; /* R10: an empty slot takes no part in the min */
    }
    return o->M[i];
}

static void recompute_node(orc_per *o, uint64_t i)
{
    o->S[i] = node_sum(o, 2 * i) + node_sum(o, 2 * i + 1);
    float a = node_min(o, 2 * i), b = node_min(o, 2 * i + 1);
    o->M[i] = a < b ? a : b;
}

/* Per-element leaf-to-root propagation: O(log n) per changed leaf. */
static void propagate_leaf(orc_per *o, uint64_t leaf)
{
    for (uint64_t i = (leaf + o->n) >> 1; i >= 1; i >>= 1)
        recompute_node(o, i);
}

/* Bottom-up rebuild of every internal node, a level finishing before the one above it
 * [SEG "Second Port"]: descending node index visits children before parents. */
static void rebuild_all(orc_per *o)
{
    for (uint64_t i = o->n - 1; i >= 1; --i)
        recompute_node(o, i);
}

/* ------------------------------------------------------------------------------------------
 * Priority transforms [GPR "Priority update", "Error Handling & Fallback"], readings R2-R3.
 * ------------------------------------------------------------------------------------------ */
static float raw_from_td(float td, double eps, float max_at_start)
{
    if (isnan(td))
        return (float)eps;
    float a = fabsf(td);
    if (isinf(a))
        return max_at_start;
    return (float)((double)a + eps);
}

static float raw_from_priority(float p, double eps, float max_at_start)
{
    if (isnan(p))
        return (float)eps;
    if (isinf(p) && p > 0.0f)
        return max_at_start;
    if ((double)p < eps)
        return (float)eps;
    return p;
}

static float leaf_from_raw(float raw, double alpha)
{
    return (float)pow((double)raw, alpha);
}

/* ------------------------------------------------------------------------------------------ */

orc_per *orc_create(uint64_t capacity, uint32_t state_dim, uint32_t row_stride_out,
                    double alpha, double eps, uint32_t mode, uint64_t seed, int with_ring)
{
    if (capacity == 0 || capacity > (1ull << 40) || row_stride_out < state_dim)
        return NULL;
    if (!(eps > 0.0) || !(alpha >= 0.0) || mode > ORC_FLAT)
        return NULL;
    orc_per *o = (orc_per *)calloc(1, sizeof(orc_per));
    if (!o)
        return NULL;
    o->capacity = capacity;
    o->n = 1;
    while (o->n < capacity)
        o->n <<= 1;
    o->d = state_dim;
    o->dp = row_stride_out;
    o->alpha = alpha;
    o->eps = eps;
    o->mode = mode;
    o->seed = seed;
    o->with_ring = with_ring;
    o->max_raw = 1.0f; /* R4 */
    int ok = 1;
    if (mode == ORC_PROPORTIONAL) {
        o->L = (float *)calloc(o->n, sizeof(float));
        o->S = (double *)calloc(o->n, sizeof(double));
        o->M = (float *)calloc(o->n, sizeof(float));
        ok = o->L && o->S && o->M;
        if (ok)
            rebuild_all(o);
    } else if (mode == ORC_FLAT) {
        o->L = (float *)calloc(o->n, sizeof(float));
        ok = o->L != NULL;
    } else if (mode == ORC_RANK) {
        o->raw = (float *)calloc(capacity, sizeof(float));
        o->cdf = (double *)calloc(capacity + 1, sizeof(double));
        ok = o->raw && o->cdf;
        if (ok) {
            /* cdf[r] = sum_{k<=r} k^-alpha, compensated (Kahan) summation in binary64 */
            double sum = 0.0, comp = 0.0;
            o->cdf[0] = 0.0;
            for (uint64_t k = 1; k <= capacity; ++k) {
                double term = pow((double)k, -alpha);
                double y = term - comp;
                double t = sum + y;
                comp = (t - sum) - y;
                sum = t;
                o->cdf[k] = sum;
            }
        }
    }
    if (ok && with_ring && state_dim > 0) {
        o->states = (float *)calloc(capacity * state_dim, sizeof(float));
        o->next = (float *)calloc(capacity * state_dim, sizeof(float));
        ok = o->states && o->next;
    }
    if (ok && with_ring) {
        o->actions = (uint32_t *)calloc(capacity, sizeof(uint32_t));
        o->rewards = (float *)calloc(capacity, sizeof(float));
        o->dones = (uint8_t *)calloc(capacity, sizeof(uint8_t));
        ok = o->actions && o->rewards && o->dones;
    }
    if (!ok) {
        orc_destroy(o);
        return NULL;
    }
    return o;
}

void orc_destroy(orc_per *o)
{
    if (!o)
        return;
    free(o->L);
    free(o->S);
    free(o->M);
    free(o->raw);
    free(o->cdf);
    free(o->states);
    free(o->next);
    free(o->actions);
    free(o->rewards);
    free(o->dones);
    free(o);
}

/* [GPR "Experience Insertion"]: row k goes to slot (cursor + k) mod capacity, in order, so a
 * later k wins a slot when count > capacity; new rows get the running maximum priority unless
 * the caller gives one. */
int orc_add(orc_per *o, uint64_t count, const float *states, const float *next_states,
            const uint32_t *actions, const float *rewards, const uint8_t *dones,
            const float *raw_prio)
{
    if (!o)
        return ORC_EINVAL;
    if (o->with_ring && count > 0 && (!actions || !rewards || !dones))
        return ORC_EINVAL;
    if (o->with_ring && o->d > 0 && count > 0 && (!states || !next_states))
        return ORC_EINVAL;
    float max_at_start = o->max_raw;
    int bulk = (o->mode == ORC_PROPORTIONAL) && (count * 8 >= o->n);
    for (uint64_t k = 0; k < count; ++k) {
        uint64_t slot = (o->cursor + k) % o->capacity;
        float raw = raw_prio ? raw_from_priority(raw_prio[k], o->eps, max_at_start) : max_at_start;
        if (o->with_ring) {
            if (o->d > 0) {
                memcpy(o->states + slot * o->d, states + k * o->d, o->d * sizeof(float));
                memcpy(o->next + slot * o->d, next_states + k * o->d, o->d * sizeof(float));
            }
            o->actions[slot] = actions[k];
            o->rewards[slot] = rewards[k];
            o->dones[slot] = dones[k];
        }
        if (o->mode == ORC_PROPORTIONAL) {
            o->L[slot] = leaf_from_raw(raw, o->alpha);
            if (!bulk)
                propagate_leaf(o, slot);
        } else if (o->mode == ORC_FLAT) {
            o->L[slot] = leaf_from_raw(raw, o->alpha);
        } else if (o->mode == ORC_RANK) {
            o->raw[slot] = raw;
        }
        if (raw > o->max_raw)
            o->max_raw = raw;
    }
    if (bulk)
        rebuild_all(o);
    o->cursor = (o->cursor + count) % o->capacity;
    o->size = o->size + count < o->capacity ? o->size + count : o->capacity;
    return ORC_OK;
}

/* [SEG "Sampling Is a Descent"]: walk from the root; go left when the left child's sum exceeds
 * the remaining mass, otherwise subtract it and go right. */
/* R26: the cumulative array of the filled slots, summed left to right in binary64 */
static double *flat_cumulative(const orc_per *o)
{
    double *C = (double *)malloc((o->size ? o->size : 1) * sizeof(double));
    if (!C)
        return NULL;
    double acc = 0.0;
    for (uint64_t i = 0; i < o->size; ++i) {
        acc += (double)o->L[i];
        C[i] = acc;
    }
    return C;
}

/* R26 with R6: the first i in [0, s) with C[i] > mass, or s when there is none */
static uint64_t flat_search(const double *C, uint64_t s, double mass)
{
    uint64_t lo = 0, hi = s;
    while (lo < hi) {
        uint64_t mid = lo + (hi - lo) / 2;
        if (C[mid] > mass)
            hi = mid;
        else
            lo = mid + 1;
    }
    return lo;
}

int64_t orc_descend(const orc_per *o, double mass, double *rem)
{
    if (o->mode == ORC_FLAT) { /* flat mode locates the mass in the cumulative array */
        double *C = flat_cumulative(o);
        if (!C || o->size == 0) {
            free(C);
            return -1;
        }
        uint64_t i = flat_search(C, o->size, mass);
        if (rem)
            *rem = mass - (i == 0 ? 0.0 : C[i - 1]);
        free(C);
        return (int64_t)i;
    }
    if (o->mode != ORC_PROPORTIONAL) /* the descent needs the tree */
        return -1;
    uint64_t idx = 1;
    while (idx < o->n) {
        double left = node_sum(o, 2 * idx);
        if (left > mass) {
            idx = 2 * idx;
        } else {
            mass -= left;
            idx = 2 * idx + 1;
        }
    }
    if (rem)
        *rem = mass;
    return (int64_t)(idx - o->n);
}

typedef struct {
    float key;
    uint32_t idx;
} rank_pair;

static int rank_cmp(const void *pa, const void *pb)
{
    const rank_pair *a = (const rank_pair *)pa, *b = (const rank_pair *)pb;
    if (a->key > b->key)
        return -1;
    if (a->key < b->key)
        return 1;
    return a->idx < b->idx ? -1 : (a->idx > b->idx ? 1 : 0);
}

int64_t orc_rank_order(const orc_per *o, uint32_t *sorted_idx)
{
    if (!o || o->mode != ORC_RANK)
        return ORC_EINVAL;
    uint64_t s = o->size;
    rank_pair *pairs = (rank_pair *)malloc((s ? s : 1) * sizeof(rank_pair));
    if (!pairs)
        return ORC_ENOMEM;
    for (uint64_t i = 0; i < s; ++i) {
        pairs[i].key = o->raw[i];
        pairs[i].idx = (uint32_t)i;
    }
    /* (key descending, index ascending) is a total order, so any sort gives the stable
     * descending order [GPR "Rank-based" step 1]. */
    qsort(pairs, s, sizeof(rank_pair), rank_cmp);
    for (uint64_t i = 0; i < s; ++i)
        sorted_idx[i] = pairs[i].idx;
    free(pairs);
    return (int64_t)s;
}

static void gather_row(const orc_per *o, uint32_t j, uint64_t slot, float *out_states,
                       float *out_next, uint32_t *out_actions, float *out_rewards,
                       uint8_t *out_dones)
{
    /* [GPR "Sampling Kernels" step 4]; padded rows as in "True Single-Graph Implementation
     * Plan", Task 2 (gather_f32_rows_padded): columns past state_dim are 0. */
    for (uint32_t c = 0; c < o->dp; ++c) {
        if (out_states)
            out_states[(uint64_t)j * o->dp + c] = c < o->d ? o->states[slot * o->d + c] : 0.0f;
        if (out_next)
            out_next[(uint64_t)j * o->dp + c] = c < o->d ? o->next[slot * o->d + c] : 0.0f;
    }
    if (out_actions)
        out_actions[j] = o->actions[slot];
    if (out_rewards)
        out_rewards[j] = o->rewards[slot];
    if (out_dones)
        out_dones[j] = o->dones[slot];
}

/* ------------------------------------------------------------------------------------------
 * Locating one draw.  Every mode maps a mass m in [0, T) to the slot whose extent
 * [C(i-1), C(i)) holds it (R6): the tree by the descent, flat mode by a search of the
 * cumulative array, uniform mode by a division, rank mode by a search of the CDF (then the slot
 * of that rank).  The draw lies near a boundary -- the parity bar's excuse for an index
 * mismatch -- when it fell off the end (R7) or when its mass is within 1e-6 * T of either end
 * of the extent: m - C(i-1) < 1e-6 T or C(i) - m < 1e-6 T.
 * ------------------------------------------------------------------------------------------ */

/* Test builds only: ORC_PLANT = 1..4 plants one known mistake in the near-boundary rule, so a
 * test can show that the rule's pins catch it (1: an absolute tolerance of 1e-6; 2: a fall-off
 * not counted; 3: the tree's upper distance taken against the next leaf; 4: the upper end not
 * tested).  The oracle proper is built with ORC_PLANT = 0. */
#ifndef ORC_PLANT
#define ORC_PLANT 0
#endif

typedef struct {
    double T;        /* the call's total */
    double *C;       /* flat mode: cumulative array of the filled slots */
    uint32_t *order; /* rank mode: slots by rank */
} locate_ctx;

static int locate_begin(const orc_per *o, locate_ctx *c)
{
    c->C = NULL;
    c->order = NULL;
    if (o->mode == ORC_PROPORTIONAL) {
        c->T = node_sum(o, 1);
    } else if (o->mode == ORC_FLAT) {
        c->C = flat_cumulative(o);
        if (!c->C)
            return ORC_ENOMEM;
        c->T = c->C[o->size - 1];
    } else if (o->mode == ORC_UNIFORM) {
        c->T = (double)o->size;
    } else {
        c->order = (uint32_t *)malloc(o->size * sizeof(uint32_t));
        if (!c->order)
            return ORC_ENOMEM;
        orc_rank_order(o, c->order);
        c->T = o->cdf[o->size];
    }
    return ORC_OK;
}

static void locate_end(locate_ctx *c)
{
    free(c->C);
    free(c->order);
}

/* below = m - C(i-1), above = C(i) - m */
static int near_boundary(int fell_off, double below, double above, double T)
{
    double tol = 1e-6 * T;
#if ORC_PLANT == 1
    tol = 1e-6;
#elif ORC_PLANT == 2
    fell_off = 0;
#elif ORC_PLANT == 4
    above = INFINITY;
#endif
    return fell_off || below < tol || above < tol;
}

/* The slot of one mass; *rank (rank mode) the rank, *rem the mass above the extent's start,
 * *near the boundary flag. */
static uint64_t locate(const orc_per *o, const locate_ctx *c, double mass, uint64_t *rank,
                       double *rem, int *near)
{
    uint64_t s = o->size, slot = 0;
    int fell_off = 0;
    double below = 0.0, above = 0.0;
    if (o->mode == ORC_PROPORTIONAL) {
        double r = 0.0;
        int64_t leaf = orc_descend(o, mass, &r);
        if ((uint64_t)leaf >= s) { /* R7 */
            leaf = (int64_t)s - 1;
            fell_off = 1;
        }
        slot = (uint64_t)leaf;
        below = r;
        above = (double)o->L[slot] - r;
#if ORC_PLANT == 3
        if (slot + 1 < o->n)
            above = (double)o->L[slot + 1] - r;
#endif
    } else if (o->mode == ORC_FLAT) {
        /* R26: the first entry of the cumulative array above the mass */
        slot = flat_search(c->C, s, mass);
        if (slot >= s) {
            slot = s - 1;
            fell_off = 1;
        }
        below = mass - (slot ? c->C[slot - 1] : 0.0);
        above = c->C[slot] - mass;
    } else if (o->mode == ORC_UNIFORM) {
        /* R24: every filled slot weighs 1, so the walk is a division */
        double fl = floor(mass);
        slot = (uint64_t)fl;
        if (slot >= s) {
            slot = s - 1;
            fell_off = 1;
        }
        below = mass - fl;
        above = 1.0 - below;
    } else {
        /* smallest r in [1, s] with cdf[r] > mass (binary search over the CDF) */
        uint64_t lo = 1, hi = s + 1;
        while (lo < hi) {
            uint64_t mid = lo + (hi - lo) / 2;
            if (o->cdf[mid] > mass)
                hi = mid;
            else
                lo = mid + 1;
        }
        uint64_t r = lo;
        if (r > s) {
            r = s;
            fell_off = 1;
        }
        slot = c->order[r - 1];
        below = mass - o->cdf[r - 1];
        above = o->cdf[r] - mass;
        *rank = r;
    }
    *rem = below;
    *near = near_boundary(fell_off, below, above, c->T);
    return slot;
}

int orc_locate(const orc_per *o, double mass, int64_t *slot, double *rem, uint8_t *near)
{
    if (!o || !slot || o->size == 0)
        return o && o->size == 0 ? ORC_EEMPTY : ORC_EINVAL;
    locate_ctx c;
    if (locate_begin(o, &c) != ORC_OK)
        return ORC_ENOMEM;
    uint64_t r = 0;
    double left = 0.0;
    int nb = 0;
    *slot = (int64_t)locate(o, &c, mass, &r, &left, &nb);
    if (rem)
        *rem = left;
    if (near)
        *near = (uint8_t)nb;
    locate_end(&c);
    return ORC_OK;
}

int orc_sample(orc_per *o, uint32_t B, float beta, int64_t *idx, float *w, float *out_states,
               float *out_next, uint32_t *out_actions, float *out_rewards, uint8_t *out_dones,
               uint8_t *near, double *rem, double *mass_out)
{
    if (!o || !idx || B == 0)
        return ORC_EINVAL;
    if (!o->with_ring && (out_states || out_next || out_actions || out_rewards || out_dones))
        return ORC_EINVAL;
    if (o->size == 0)
        return ORC_EEMPTY;
    uint64_t call = o->calls;
    locate_ctx c;
    if (locate_begin(o, &c) != ORC_OK)
        return ORC_ENOMEM;
    /* p_min (R8): the min tree's root, or the smallest filled leaf without a tree */
    float pmin = INFINITY;
    if (o->mode == ORC_PROPORTIONAL) {
        pmin = node_min(o, 1);
    } else if (o->mode == ORC_FLAT) {
        for (uint64_t i = 0; i < o->size; ++i)
            if (o->L[i] < pmin)
                pmin = o->L[i];
    }
    /* counter tags: 0 proportional and flat (the same draws), 1 rank, 2 uniform */
    uint32_t tag = o->mode == ORC_RANK ? 1u : (o->mode == ORC_UNIFORM ? 2u : 0u);
    double seg = c.T / (double)B;
    for (uint32_t j = 0; j < B; ++j) {
        double u = orc_uniform53(o->seed, j, call, tag);
        double mass = ((double)j + u) * seg; /* R5 */
        uint64_t r = 0;
        double left = 0.0;
        int nb = 0;
        uint64_t slot = locate(o, &c, mass, &r, &left, &nb);
        idx[j] = (int64_t)slot;
        if (w) {
            if (o->mode == ORC_RANK) /* R11: (n P(r))^-beta / max_w = (r / n)^(alpha beta) */
                w[j] = (float)pow((double)r / (double)o->size, o->alpha * (double)beta);
            else if (o->mode == ORC_UNIFORM)
                w[j] = 1.0f;
            else /* R8 */
                w[j] = (float)pow((double)o->L[slot] / (double)pmin, -(double)beta);
        }
        if (near)
            near[j] = (uint8_t)nb;
        if (rem)
            rem[j] = left;
        if (mass_out)
            mass_out[j] = mass;
        if (o->with_ring)
            gather_row(o, j, slot, out_states, out_next, out_actions, out_rewards, out_dones);
    }
    locate_end(&c);
    o->calls = call + 1;
    return ORC_OK;
}

/* [GPR "Priority update"] with readings R2-R4, R9, R12; propagation per element. */
int orc_update(orc_per *o, uint32_t B, const int64_t *idx, const float *td)
{
    if (!o || (B > 0 && (!idx || !td)))
        return ORC_EINVAL;
    if (o->mode == ORC_UNIFORM) /* R24: no priorities */
        return 0;
    float max_at_start = o->max_raw;
    int skipped = 0;
    for (uint32_t j = 0; j < B; ++j) {
        int64_t i = idx[j];
        if (i < 0 || (uint64_t)i >= o->size) {
            ++skipped;
            continue;
        }
        float raw = raw_from_td(td[j], o->eps, max_at_start);
        if (o->mode == ORC_PROPORTIONAL) {
            o->L[i] = leaf_from_raw(raw, o->alpha);
            propagate_leaf(o, (uint64_t)i);
        } else if (o->mode == ORC_FLAT) {
            o->L[i] = leaf_from_raw(raw, o->alpha);
        } else {
            o->raw[i] = raw;
        }
        if (raw > o->max_raw)
            o->max_raw = raw;
    }
    return skipped;
}

uint64_t orc_capacity(const orc_per *o) { return o->capacity; }
uint64_t orc_nleaves(const orc_per *o) { return o->n; }
uint64_t orc_size(const orc_per *o) { return o->size; }
uint64_t orc_cursor(const orc_per *o) { return o->cursor; }
uint64_t orc_sample_calls(const orc_per *o) { return o->calls; }
float orc_max_raw(const orc_per *o) { return o->max_raw; }

double orc_total(const orc_per *o)
{
    if (o->mode == ORC_RANK)
        return o->cdf[o->size];
    if (o->mode == ORC_UNIFORM)
        return (double)o->size;
    if (o->mode == ORC_FLAT) { /* R26: the last entry of the cumulative array */
        double acc = 0.0;
        for (uint64_t i = 0; i < o->size; ++i)
            acc += (double)o->L[i];
        return acc;
    }
    return node_sum(o, 1);
}

float orc_min(const orc_per *o)
{
    if (o->mode == ORC_RANK)
        return NAN;
    if (o->mode == ORC_UNIFORM)
        return 1.0f;
    if (o->mode == ORC_FLAT) {
        float m = INFINITY;
        for (uint64_t i = 0; i < o->size; ++i)
            if (o->L[i] < m)
                m = o->L[i];
        return m;
    }
    return node_min(o, 1);
}

const float *orc_leaves(const orc_per *o) { return o->L; }
const double *orc_sums(const orc_per *o) { return o->S; }
const float *orc_mins(const orc_per *o) { return o->M; }
const float *orc_raw(const orc_per *o) { return o->raw; }
const double *orc_cdf(const orc_per *o) { return o->cdf; }
const float *orc_ring_states(const orc_per *o) { return o->states; }
const float *orc_ring_next(const orc_per *o) { return o->next; }
