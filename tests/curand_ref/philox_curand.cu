// Test infrastructure: cuRAND's device Philox4x32-10 (an independent implementation of the
// generator of Salmon et al., SC'11) evaluated at given (counter, key) pairs, to pin the
// oracle's generator.  curand_init(seed, subsequence, offset) sets key = (seed lo, seed hi) and
// counter = (offset/4 lo, offset/4 hi, subsequence lo, subsequence hi) (skipahead adds offset/4 to
// the counter's low 64 bits); with offsets in multiples of 4 the next curand4 returns the four
// output words of that counter.
#include <curand_kernel.h>

__global__ void k_philox_curand(const unsigned *ctr, const unsigned *key, unsigned *out, int n)
{
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    const unsigned long long seed = ((unsigned long long)key[2 * i + 1] << 32) | key[2 * i];
    const unsigned long long off4 = ((unsigned long long)ctr[4 * i + 1] << 32) | ctr[4 * i];
    const unsigned long long sub = ((unsigned long long)ctr[4 * i + 3] << 32) | ctr[4 * i + 2];
    curandStatePhilox4_32_10_t st;
    curand_init(seed, sub, 0ull, &st);
    // advance the low 64 counter bits by off4 (an offset of 4 per counter step) in pieces whose
    // offsets fit 64 bits
    for (int r = 0; r < 8; ++r) skipahead(4ull * (off4 >> 3), &st);
    skipahead(4ull * (off4 & 7ull), &st);
    const uint4 v = curand4(&st);
    out[4 * i] = v.x;
    out[4 * i + 1] = v.y;
    out[4 * i + 2] = v.z;
    out[4 * i + 3] = v.w;
}

extern "C" int philox_curand(const unsigned *d_ctr, const unsigned *d_key, unsigned *d_out, int n)
{
    k_philox_curand<<<(n + 127) / 128, 128>>>(d_ctr, d_key, d_out, n);
    return (int)cudaDeviceSynchronize();
}
