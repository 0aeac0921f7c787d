// Tensor-core paged decode over E4M3 pools: the variants whose E4M3
// operands hold groups of up to 4 query heads (MMA N = 16), compiled apart
// from the 8-head ones so that the two build in parallel.
#include <cuda.h>  // CUtensorMap and its enums only

#include "pa_decode_tc.cuh"

namespace pa {

TcKernel tc8_pick4(bool bf16, int D, bool span, bool compact, int *smem, int *cols) {
    return tc8_pick<4>(bf16, D, span, compact, smem, cols);
}

}  // namespace pa
