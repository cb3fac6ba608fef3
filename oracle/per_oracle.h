/*
 * per_oracle.h -- the oracle's own interface.
 *
 * TEST INFRASTRUCTURE ONLY.  The oracle is a plain, slow, sequential CPU implementation of
 * GPU-resident prioritized experience replay.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg load it.  It shares no code, header, table or helper with the
 * CUDA library; the two meet only through seeded inputs produced elsewhere.
 *
 * Every floating-point step is plain IEEE-754 binary64 (or binary32 where the method stores
 * binary32), evaluated in the order written, with contraction disabled at build time.
 */
#ifndef PER_ORACLE_H
#define PER_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORC_PROPORTIONAL = 0, ORC_RANK = 1, ORC_UNIFORM = 2, ORC_FLAT = 3 };
enum { ORC_OK = 0, ORC_EINVAL = -1, ORC_EEMPTY = -2, ORC_ENOMEM = -3 };

typedef struct orc_per orc_per;

/* Philox4x32-10 of Salmon et al. (SC'11): ten rounds of the two-multiplier S-box with the
 * published multipliers and Weyl key increments.  ctr[4], key[2] in; out[4] out. */
void orc_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]);

/* The uniform u in [0,1) that draw j of sample call `call` uses: counter (j, call lo, call hi,
 * tag), key (seed lo, seed hi); u = ((x0 << 21) | (x1 >> 11)) * 2^-53, exact in binary64. */
double orc_uniform53(uint64_t seed, uint32_t j, uint64_t call, uint32_t tag);

/* Create a replay buffer of `capacity` slots, rows of `state_dim` floats gathered into rows of
 * `row_stride_out` floats.  with_ring = 0 keeps only the priority structures (no row
 * mirror): sampling then returns indices and weights only. */
orc_per *orc_create(uint64_t capacity, uint32_t state_dim, uint32_t row_stride_out,
                    double alpha, double eps, uint32_t mode, uint64_t seed, int with_ring);
void orc_destroy(orc_per *o);

/* Insert `count` transitions at the ring cursor.  raw_prio may be NULL (every new row gets the
 * running maximum raw priority).  Any array may be NULL when with_ring = 0. */
int orc_add(orc_per *o, uint64_t count, const float *states, const float *next_states,
            const uint32_t *actions, const float *rewards, const uint8_t *dones,
            const float *raw_prio);

/* Draw a stratified batch of B.  Outputs other than idx may be NULL.  near[j] = 1 marks a
 * draw whose mass lies within 1e-6 * total of a boundary of the chosen leaf (or fell off the
 * end); rem[j] is the mass left when the descent reached the leaf (rank mode: mass minus the
 * CDF below the chosen rank); mass[j] the draw's mass. */
int orc_sample(orc_per *o, uint32_t B, float beta, int64_t *idx, float *w, float *out_states,
               float *out_next, uint32_t *out_actions, float *out_rewards, uint8_t *out_dones,
               uint8_t *near, double *rem, double *mass);

/* Where one mass lands, by the same step orc_sample takes for each draw (every mode): *slot
 * the chosen slot (after clamping), *rem the mass above the start of its extent, *near the
 * near-boundary flag.  rem and near may be NULL.  ORC_EEMPTY when no slot is filled. */
int orc_locate(const orc_per *o, double mass, int64_t *slot, double *rem, uint8_t *near);

/* Scatter new priorities from TD errors.  Returns the number of skipped entries (index outside
 * the filled slots) or a negative error. */
int orc_update(orc_per *o, uint32_t B, const int64_t *idx, const float *td);

/* The descent of a single mass (proportional mode).  *rem receives the mass left at the leaf.
 * Returns the leaf before any clamping. */
int64_t orc_descend(const orc_per *o, double mass, double *rem);

/* Rank mode: indices of the filled slots sorted by raw priority descending, ties by index
 * ascending.  sorted_idx has room for size entries.  Returns size. */
int64_t orc_rank_order(const orc_per *o, uint32_t *sorted_idx);

/* Accessors (pointers stay owned by the oracle). */
uint64_t orc_capacity(const orc_per *o);
uint64_t orc_nleaves(const orc_per *o); /* power of two >= capacity */
uint64_t orc_size(const orc_per *o);
uint64_t orc_cursor(const orc_per *o);
uint64_t orc_sample_calls(const orc_per *o);
float orc_max_raw(const orc_per *o);
double orc_total(const orc_per *o); /* proportional: root sum; rank: CDF at size */
float orc_min(const orc_per *o);    /* proportional: root of the min tree */
const float *orc_leaves(const orc_per *o);  /* [nleaves] p^alpha, 0 = empty slot */
const double *orc_sums(const orc_per *o);   /* [nleaves], entry 0 unused */
const float *orc_mins(const orc_per *o);    /* [nleaves], entry 0 unused */
const float *orc_raw(const orc_per *o);     /* rank mode: [capacity] raw priorities */
const double *orc_cdf(const orc_per *o);    /* rank mode: [capacity + 1], cdf[0] = 0 */
const float *orc_ring_states(const orc_per *o);
const float *orc_ring_next(const orc_per *o);

#ifdef __cplusplus
}
#endif
#endif
