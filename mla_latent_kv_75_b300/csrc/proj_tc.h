// Arguments of the tensor-core projection GEMM (gemm_tc.cu).
#pragma once
#include <stdint.h>

namespace mla {

// Y[n, o] = sum_k W[o, k] X[n, k] with W = [W0 (O0 rows); W1 (O1 rows); W2 (O2 rows)], K input
// columns. W1 and W2 are optional; when W2 is set, W1 is padded to whole 128-row tiles and W2's
// rows start at output row 128 * (O0 / 128 + ceil(O1 / 128)). X2, if set, is a second bf16
// operand accumulated against the same W (hi/lo split inputs).
struct ProjArgs {
  const void* W0;
  int O0;
  const void* W1;
  int O1;
  const void* W2;
  int O2;
  int K;
  const void* X;
  const void* X2;
  int64_t ldx;
  int N;
  int kid;
};

}  // namespace mla
