/*
 * gbper.h -- GPU-resident prioritized experience replay (PER) on one GB300 (sm_103a).
 *
 * A C ABI over plain pointers and sizes.  Every transition, priority and batch lives in device
 * memory; the library owns the replay ring and the priority trees, the caller owns every input
 * and output buffer it passes.  No call takes or returns a torch type.
 *
 * Sources (cited by page title and section):
 *   "GPU-Resident Prioritized Experience Replay" (foxhunt design document): Architecture,
 *     Sampling Kernels (Proportional, Rank-based), Priority update, Experience Insertion,
 *     Error Handling & Fallback.
 *   "Putting prioritized replay's segment tree on a GPU": The Tree Under Every Prioritized
 *     Replay, Sampling Is a Descent, Second Port: Make the Update GPU-Shaped.
 *   "True Single-Graph Implementation Plan": Task 2 (padded row gather, int64 indices),
 *     Task 3 (gather straight into the trainer's buffers), Task 4 (device-side counters),
 *     Task 5 (PER calls as stream work that a CUDA graph can capture).
 *
 * Conventions shared by every call
 *   - Streams.  `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *     stream).  Work is enqueued on it; no call below synchronises the host unless its
 *     comment says so (per_total, per_min, per_status_device, per_read_state).
 *   - Device pointers.  Arguments named d_* are device addresses (cudaMalloc or the caching
 *     allocator of a framework) on the device that was current at per_create.  They must stay
 *     valid until the enqueued work has run.  Row arrays must be 4-byte aligned; 16-byte
 *     alignment together with a row length that is a multiple of 4 floats enables the
 *     vectorised copy paths.
 *   - Errors.  Every call returns a per_status.  Invalid host-side arguments return
 *     PER_ERR_INVALID_ARG before anything is enqueued.  A failed CUDA call returns
 *     PER_ERR_CUDA; per_last_error() then describes it.  Conditions only the device can see
 *     (an update index outside the filled slots, a bounded wait that ran out) never trap or
 *     abort: the kernel skips the offending element and sets a bit in the device error word,
 *     which per_status_device() reads and clears.  Nothing falls back to the CPU.
 *   - Concurrency.  One handle is driven from one host thread at a time, and its calls are
 *     ordered by the caller (one stream, or explicit events across streams).
 */
#ifndef GBPER_H
#define GBPER_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct per_buffer per_buffer; /* opaque; owned by the library */

typedef enum {
    PER_OK = 0,
    PER_ERR_INVALID_ARG = 1, /* rejected on the host; nothing was enqueued */
    PER_ERR_OOM = 2,         /* device allocation in per_create failed */
    PER_ERR_CUDA = 3,        /* a CUDA runtime call failed; see per_last_error */
    PER_ERR_EMPTY = 4,       /* per_sample / per_min on a buffer with no filled slot */
    PER_ERR_DEVICE_FLAG = 5, /* per_status_device: the device error word was non-zero */
    PER_ERR_TIMEOUT = 6      /* a bounded device-side wait gave up (reported as a flag bit) */
} per_status;

/* Sampling modes ("GPU-Resident Prioritized Experience Replay", Sampling Kernels). */
enum {
    PER_MODE_PROPORTIONAL = 0, /* P(i) = p_i^alpha / sum_k p_k^alpha, sum tree + min tree */
    PER_MODE_RANK = 1,         /* P(i) proportional to 1 / rank(i)^alpha, rank by raw priority */
    PER_MODE_UNIFORM = 2,      /* P(i) = 1 / size: the plain replay PER replaces; priorities unused */
    PER_MODE_FLAT = 3          /* proportional, located by the pages' own flat design: an inclusive
                                  sum of the leaves rebuilt at each sample and a search per draw
                                  ("Sampling Kernels", Proportional steps 2-3); no tree */
};

/* Bits of the device error word (per_status_device). */
enum {
    PER_DEVFLAG_BAD_INDEX = 1u, /* an update named an index outside [0, size); it was skipped */
    PER_DEVFLAG_TIMEOUT = 2u,   /* a bounded wait gave up; the call's results are not valid */
    PER_DEVFLAG_RANK_STALE = 4u /* rank mode: more slots were written between two samples than the
                                   order merge can take (only reachable by replaying a captured
                                   sample after more writes than at capture); the order is stale */
};

/* per_config.flags */
enum {
    PER_FLAG_RANK_RESORT = 1u, /* rank mode: sort every filled slot at each sample instead of
                                  merging the slots written since the previous one (same order) */
    PER_FLAG_DONES_F32 = 2u    /* per_sample writes dones as float 0.0f / 1.0f (d_dones is float*,
                                  4-byte aligned), the trainer's format ("True Single-Graph
                                  Implementation Plan", Task 3) */
};

typedef struct {
    double alpha;            /* priority exponent, >= 0 */
    double eps;              /* added to |td| before the exponent; > 0 */
    uint32_t mode;           /* PER_MODE_* */
    uint32_t row_stride_out; /* floats per gathered state row, >= state_dim (0: state_dim);
                                columns past state_dim are written as 0.0f */
    uint64_t seed;           /* key of the Philox4x32-10 stream that draws the batches */
    uint32_t flags;          /* PER_FLAG_* bits; others must be 0 */
    uint32_t rebuild_batch;  /* update batches of at least this many entries scatter their
                                priorities and rebuild every tree level instead of climbing from
                                each changed leaf (same result); 0: the crossover measured on
                                GB300 (max(leaves / 128, 1024) proportional; rank mode
                                always scatters), and smaller batches too while recent
                                updates crowded a subtree (see per_update_priorities);
                                UINT32_MAX: never; any other value: from that size, with
                                no regard to crowding */
    uint32_t element_batch;  /* proportional mode: update batches of fewer entries than this
                                propagate entry by entry, each from its leaf to the root (same
                                result); 0: the crossover measured on GB300 (3: batches of
                                one or two entries); 1: never; UINT32_MAX: always */
    uint32_t reserved;       /* 0 */
} per_config;

/*
 * per_create -- allocate a replay buffer of `capacity` slots holding rows of `state_dim`
 * floats ("GPU-Resident Prioritized Experience Replay", Architecture: a fixed-capacity ring
 * of states, next_states, actions, rewards, dones and priorities; no allocation during
 * training).  Proportional mode also allocates the sum tree (binary64 internal nodes over
 * binary32 leaves p^alpha) and its twin min tree ("Putting prioritized replay's segment tree
 * on a GPU", The Tree Under Every Prioritized Replay); the tree has the next power of two
 * >= capacity leaves, and the extra leaves are never filled.  Rank mode allocates the raw
 * priorities, the sort workspace and the rank CDF, which it computes here.
 * Every later call reuses these allocations.  The device current at this call owns them.
 *   capacity  1 .. 2^31 slots.
 *   state_dim floats per state row, 0 .. 65536.
 *   cfg       copied; NULL means alpha 0.6, eps 1e-6, proportional, stride = state_dim.
 *   out       receives the handle (unchanged on error).
 * Errors: PER_ERR_INVALID_ARG (bad sizes or config), PER_ERR_OOM, PER_ERR_CUDA.
 */
per_status per_create(uint64_t capacity, uint32_t state_dim, const per_config *cfg,
                      per_buffer **out);

/* per_destroy -- synchronise the device, release every allocation and the handle.
 * NULL is accepted and ignored. */
per_status per_destroy(per_buffer *h);

/*
 * per_add -- insert `count` transitions at the ring cursor ("GPU-Resident Prioritized
 * Experience Replay", Experience Insertion): row k goes to slot (cursor + k) mod capacity, so
 * when count > capacity only the last `capacity` rows stay; the cursor wraps and the filled
 * size grows to at most capacity.  Each new slot's raw priority is d_raw_prio[k] or, when
 * d_raw_prio is NULL, the running maximum raw priority ("new experiences get max_priority").
 * Raw priorities pass the clamp of Error Handling & Fallback: NaN becomes eps, +Inf becomes
 * the running maximum as it stood when the call began, values below eps become eps.  The
 * running maximum then takes every new raw priority.  Proportional mode writes the leaves
 * p^alpha (binary64 pow rounded to binary32) and rebuilds the dirty ancestors of both trees
 * level by level ("Putting prioritized replay's segment tree on a GPU", Second Port).
 *   d_states, d_next  [count x state_dim] float, row-major (may be NULL when state_dim = 0).
 *   d_actions [count] uint32, d_rewards [count] float, d_dones [count] uint8.
 *   d_raw_prio [count] float or NULL.
 * count = 0 is a no-op.  No host synchronisation.
 */
per_status per_add(per_buffer *h, uint64_t count, const float *d_states, const float *d_next,
                   const uint32_t *d_actions, const float *d_rewards, const uint8_t *d_dones,
                   const float *d_raw_prio, void *stream);

/*
 * per_sample -- draw a stratified batch of B transitions and gather it into caller buffers.
 * Proportional mode ("GPU-Resident Prioritized Experience Replay", Sampling Kernels,
 * Proportional; "Putting prioritized replay's segment tree on a GPU", Sampling Is a Descent):
 * draw j takes u_j from Philox4x32-10 (counter = (j, call lo, call hi, 0), key = seed, 53-bit
 * uniform from the first two words), mass_j = (j + u_j) * (T / B) with T the root sum, and
 * walks from the root: left when the left child's sum exceeds the mass, otherwise subtract
 * and go right.  A walk that ends past the filled slots is clamped to the last filled slot.
 * The IS weight is w = (n P(i))^-beta / max_w with max_w from the min tree, which equals
 * (p_i^alpha / p_min^alpha)^-beta.
 * Rank mode ("Sampling Kernels", Rank-based): sorts the filled slots by raw priority
 * descending (ties by slot ascending), draws mass_j = (j + u_j) * (c_size / B) with counter
 * tag 1, takes the rank r whose CDF interval c_{r-1} <= mass < c_r holds it, with
 * c_r = sum_{k<=r} k^-alpha, and weights w = (r / size)^(alpha * beta).  The order is kept
 * between calls: when it exists and at most 4096 slots (and at most an eighth of the filled
 * ones, by the host's count of inserted and updated entries) were written since, only those
 * slots are merged back into it; otherwise every filled slot is sorted again.  Both give the
 * same order.
 * Uniform mode (the plain replay that PER replaces, "GPU-Resident Prioritized Experience
 * Replay", Experience Insertion): every filled slot weighs 1, so draw j (counter tag 2) takes
 * mass_j = (j + u_j) * (size / B) and slot floor(mass_j), clamped to the last filled slot;
 * w = 1.
 * Flat mode ("Sampling Kernels", Proportional steps 2-5, the pages' own design): the same draws
 * as proportional mode (tag 0); the call first sums the filled leaves into the inclusive array
 * C[i] = L[0] + ... + L[i] (fixed-point sums with the unit 2^-52 of the largest leaf's binade,
 * each prefix rounded once to binary64), then draw j takes the first slot with
 * C[slot] > mass_j, T = C[size-1], and the same weight with p_min the smallest filled leaf.
 * The sums round differently from the tree's, so slot choices can differ from proportional
 * mode only for masses within rounding distance of a boundary.  Flat mode needs alpha <= 1.
 * Gather ("True Single-Graph Implementation Plan", Task 2/3): row j of d_states and d_next
 * receives the chosen slot's row, padded with 0.0f to row_stride_out floats.
 *   d_idx [B] int64 (required); d_w [B] float; d_states, d_next [B x row_stride_out] float;
 *   d_actions [B] uint32; d_rewards [B] float; d_dones [B] uint8 (float with
 *   PER_FLAG_DONES_F32) -- each may be NULL to skip.
 *   B in 1 .. 2^24.  beta >= 0.
 * The call counter lives on the device, so each call, captured in a graph or not, draws a
 * fresh batch.  PER_ERR_EMPTY when the buffer holds no transition (host-side count).  In rank
 * mode the slot order's length is fixed at launch, so a call made during stream capture while
 * the buffer is not yet full is refused (PER_ERR_INVALID_ARG): capture rank-mode rounds once the
 * ring is full.
 */
per_status per_sample(per_buffer *h, uint32_t B, float beta, int64_t *d_idx, float *d_w,
                      float *d_states, float *d_next, uint32_t *d_actions, float *d_rewards,
                      uint8_t *d_dones, void *stream);

/*
 * per_update_priorities -- write new priorities for a batch from its TD errors
 * ("GPU-Resident Prioritized Experience Replay", Priority update and Error Handling &
 * Fallback): raw = fl32(|td| + eps), NaN -> eps, +-Inf -> the running maximum as it stood
 * when the call began; the leaf becomes raw^alpha.  When an index repeats, the highest batch
 * position wins.  Proportional mode then rebuilds the dirty ancestors of the sum and min
 * trees level by level ("Putting prioritized replay's segment tree on a GPU", Second Port),
 * restricted to the nodes above a changed leaf.  Batches of at least per_config.rebuild_batch
 * entries instead mark each slot's last batch position in a winner word, write the winners and
 * rebuild every level of both trees (the post's level-synchronous rebuild, Measuring the
 * Trade Honestly: O(k + n) beats O(k log n) once k is a large share of n); the trees come out
 * the same.  Smaller batches climb, each warp serving one subtree's entries 32 distinct leaves at
 * a time, one group after the other, so crowding matters: the update kernels report the most
 * entries one subtree received (with the split they used) through mapped host memory, without a
 * synchronisation and a few calls late, and on each new report the next climbs split the tree
 * twice as finely when a subtree held more than 32 entries (up to 2^10 subtrees) and once as
 * coarsely again at 8 or fewer; when even the finest split leaves at least
 * 32 max(2, 5/6 leaves / 2^20) entries in a subtree, the next calls rebuild every level (measured on GB300 at 2^21 leaves,
 * B = 512: up to 465 entries in one subtree climbed in 68-104 us, rebuilt in 33 us), until the
 * counts the rebuild keeps fall below it.  PER_STATE_COUNTERS[4] reads the latest report.  A
 * rebuild_batch other than 0 keeps the size rule alone.  Flat mode writes the leaves only (scatter path
 * always; the next sample sums them).  Rank mode stores raw.  Uniform mode has no
 * priorities: the call checks its arguments and changes nothing.  The running maximum
 * takes every raw priority of the batch.  Indices outside [0, size) are skipped and set
 * PER_DEVFLAG_BAD_INDEX.
 *   d_idx [B] int64, d_td [B] float.  B in 0 .. 2^24 (0 is a no-op).
 */
per_status per_update_priorities(per_buffer *h, uint32_t B, const int64_t *d_idx,
                                 const float *d_td, void *stream);

/*
 * per_rank_refresh -- rank mode: bring the slot order up to date now, the step per_sample takes
 * first ("GPU-Resident Prioritized Experience Replay", Sampling Kernels, Rank-based step 1: the
 * filled slots sorted by raw priority descending, ties by slot ascending).  When the order exists
 * and at most 4096 slots (and at most an eighth of the filled ones) were written since it was
 * made, the written slots are merged into it; otherwise every filled slot is sorted again.  A
 * per_sample that follows with no write in between samples from this order without redoing it;
 * PER_STATE_RANK_ORDER reads it.  A buffer with no filled slot is left as it is.  No host
 * synchronisation.  As for per_sample, a call made during stream capture while the buffer is not
 * yet full is refused.
 * Errors: PER_ERR_INVALID_ARG (not rank mode, or the capture case), PER_ERR_CUDA.
 */
per_status per_rank_refresh(per_buffer *h, void *stream);

/* per_total -- the root of the sum tree (proportional), c_size (rank), size (uniform) or C[size-1]
 * after a fresh scan (flat), copied to *host_out.  Synchronises `stream`. */
per_status per_total(per_buffer *h, double *host_out, void *stream);

/* per_min -- the smallest p^alpha over filled slots: the root of the min tree (proportional) or
 * the minimum a fresh scan carries (flat); other modes are rejected.  Synchronises `stream`.
 * PER_ERR_EMPTY when no slot is filled. */
per_status per_min(per_buffer *h, float *host_out, void *stream);

/* per_size -- the number of filled slots as the host has counted the per_add calls enqueued
 * so far.  No device access.  Calls replayed from a CUDA graph are not counted here; the
 * device's own count is PER_STATE_COUNTERS[2] (per_read_state). */
per_status per_size(const per_buffer *h, uint64_t *out);

/* per_status_device -- read and clear the device error word (PER_DEVFLAG_* bits) into
 * *host_flags (may be NULL).  Synchronises `stream`.  Returns PER_ERR_DEVICE_FLAG when the
 * word was non-zero, PER_OK otherwise. */
per_status per_status_device(per_buffer *h, uint32_t *host_flags, void *stream);

/* per_last_error -- a description of the last failure on this handle ("" if none).  The
 * string stays valid until the next call on the handle.  NULL handle: the last per_create
 * failure on this thread. */
const char *per_last_error(const per_buffer *h);

/* What per_read_state copies out. */
enum {
    PER_STATE_LEAVES = 0,   /* float [nleaves]: p^alpha, 0 for empty slots (proportional) */
    PER_STATE_SUMS = 1,     /* double [nleaves]: internal sums, entry 0 unused */
    PER_STATE_MINS = 2,     /* float [nleaves]: internal mins, entry 0 unused */
    PER_STATE_RAW = 3,      /* float [capacity]: raw priorities (rank mode) */
    PER_STATE_CDF = 4,      /* double [capacity + 1]: rank CDF, entry 0 = 0 (rank mode) */
    PER_STATE_STATES = 5,   /* float [capacity x state_dim]: ring states */
    PER_STATE_NEXT = 6,     /* float [capacity x state_dim]: ring next_states */
    PER_STATE_ACTIONS = 7,  /* uint32 [capacity] */
    PER_STATE_REWARDS = 8,  /* float [capacity] */
    PER_STATE_DONES = 9,    /* uint8 [capacity] */
    PER_STATE_COUNTERS = 10, /* uint64 [5]: sample calls, cursor, size, max raw (float bits), and
                                (proportional mode) the latest update's crowding report:
                                bits 28-31 P, bits 20-27 a sequence number, bits 0-19 the
                                most entries one of its 2^P subtrees received (see
                                per_update_priorities) */
    PER_STATE_RANK_ORDER = 11, /* uint32 [size at the last sample]: slots by rank (rank mode) */
    PER_STATE_CUMULATIVE = 12  /* double [size on the device]: C[i] = leaves 0..i summed, as of the
                                  last sample, per_total or per_min (flat mode) */
};

/* per_read_state -- copy `count` elements starting at element `first` of one of the arrays
 * above into host memory at host_dst (inspection, checkpoints, tests).  Synchronises
 * `stream`.  PER_ERR_INVALID_ARG if the array does not exist in this mode or the range is
 * out of bounds. */
per_status per_read_state(per_buffer *h, uint32_t which, uint64_t first, uint64_t count,
                          void *host_dst, void *stream);

/* per_nleaves -- the tree's leaf count (power of two >= capacity). */
per_status per_nleaves(const per_buffer *h, uint64_t *out);

/*
 * per_rank_order_noalloc -- the slot order of the rank-based variant without a replay
 * buffer and without allocating: d_order[r-1] receives the slot of rank r, where rank 1 holds
 * the largest of d_raw[0, n) and equal priorities keep ascending slot order.  It runs the
 * same radix-sort kernels that per_sample uses in rank mode.  The pages have no counterpart:
 * this call exists for callers that may not allocate device memory -- code enqueuing work
 * while a CUDA graph is being captured (cudaMalloc is not permitted then), real-time loops
 * that forbid allocator latency, or hosts whose device memory belongs to another framework's
 * pool.  The call itself makes no cudaMalloc, cudaFree or other allocating call.
 *   d_raw    [n] float, device, > 0 and finite (caller-owned input).
 *   d_order  [n] uint32, device (caller-owned output).
 *   d_status one uint32, device, or NULL (caller-owned output): receives 0, or the
 *            PER_DEVFLAG_* bits of what the device met (PER_DEVFLAG_TIMEOUT: a bounded wait of
 *            the sort gave up).  The call returns before the GPU runs it, so its return value
 *            cannot carry this; read the word after the stream has reached it.
 *   n        1 .. 262144 (2^18); larger n returns PER_ERR_INVALID_ARG.
 * When a wait gave up, every entry of d_order is 0xFFFFFFFF (a value no valid slot has)
 * instead of a partial order, whether or not d_status is given.
 * Scratch: a fixed device array of about 4.3 MiB compiled into the library, which every GPU
 * that loads the library holds until the process exits.  The first call on a device looks up
 * that array's device address (cudaGetSymbolAddress) and caches it; make that first call on
 * each device before any stream capture begins.  All calls share the one array and it keeps
 * the last call's contents; every call first clears, with cudaMemsetAsync (no allocation), the
 * digit histograms, tile counters and error word that must start at zero, so a call that
 * stopped part way does not spoil the next.  Calls whose GPU work overlaps -- on different
 * streams, or concurrently from several host threads -- race on the array and must be
 * serialised by the caller.
 * Errors: PER_ERR_INVALID_ARG (NULL or misaligned pointer, n out of range), PER_ERR_CUDA.
 * It records no message for per_last_error.
 */
per_status per_rank_order_noalloc(const float *d_raw, uint32_t n, uint32_t *d_order,
                                  uint32_t *d_status, void *stream);

#ifdef __cplusplus
}
#endif
#endif
