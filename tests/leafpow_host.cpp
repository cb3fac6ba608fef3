// Host build of the binary32-power routine that the tree kernels use (leaf_pow.cuh), so that
// its error bound and its agreement with the binary64 pow can be checked without a GPU.
#include "leaf_pow.cuh"

#include <cmath>

extern "C" int lp_eval(const float *x, int n, double alpha, float *out, float *vhi, float *vlo,
                       unsigned char *fast)
{
    static const gbper::LeafPowTables tables = gbper::make_leaf_pow_tables();
    const gbper::LeafPowAlpha a = gbper::make_leaf_pow_alpha(alpha);
    for (int i = 0; i < n; ++i) {
        gbper::ff v{0.0f, 0.0f};
        float o = 0.0f;
        const bool ok = gbper::leaf_pow_fast(x[i], a, tables, &o, &v);
        fast[i] = ok ? 1 : 0;
        out[i] = ok ? o : (float)std::pow((double)x[i], alpha);
        vhi[i] = v.hi;
        vlo[i] = v.lo;
    }
    return 0;
}
