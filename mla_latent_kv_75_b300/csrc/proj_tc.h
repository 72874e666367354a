// Arguments of the tensor-core projection GEMM (gemm_tc.cu).
#pragma once
#include <stdint.h>

namespace mla {

// Y[n, o] = sum_k W[o, k] X[n, k] with W = [W0 (O0 rows); W1 (O1 rows)], K input columns.
// X2, if set, is a second bf16 operand accumulated against the same W (hi/lo split inputs).
struct ProjArgs {
  const void* W0;
  int O0;
  const void* W1;
  int O1;
  int K;
  const void* X;
  const void* X2;
  int64_t ldx;
  int N;
  int kid;
};

}  // namespace mla
