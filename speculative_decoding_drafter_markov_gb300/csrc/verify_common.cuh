// verify_common.cuh -- pieces of the verification outcome shared by the
// CUDA-core and tensor-core second phases.
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace dspark {

// [E] section 06 along the prefix: the accepted drafted tokens, then the
// correction (residual winner i_res at the first rejection; the winner i_p of
// the race over p when the residual was empty) or, all accepted, the bonus
// token i_p; the next anchor is that token.  Requests missing from the batch
// (ell < 0) get -1 everywhere.
__device__ __forceinline__ void write_outcome(const dspark_verify_args &a, const VerifyWs &w, int rq, int i_res,
                                              int i_p) {
    const int ell = w.ell[rq];
    int32_t *out = a.out_tokens + (size_t)rq * (a.gamma + 1);
    if (ell < 0) {
        a.n_accept[rq] = 0;
        for (int j = 0; j <= a.gamma; ++j) out[j] = -1;
        a.next_anchor[rq] = -1;
        return;
    }
    const int fr = w.first_rej[rq];
    const bool residual = fr < ell;
    const int n = residual ? fr : ell;
    int y = (residual && i_res >= 0) ? i_res : i_p;
    if (y < 0) {
        set_err(a.err, DSPARK_ERR_NONFINITE);
        y = 0;
    }
    a.n_accept[rq] = n;
    for (int j = 0; j <= a.gamma; ++j) out[j] = j < n ? a.x[(size_t)rq * a.gamma + j] : (j == n ? y : -1);
    a.next_anchor[rq] = y;
}

}  // namespace dspark
