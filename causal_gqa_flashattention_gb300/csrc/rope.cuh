// rope.cuh -- device helper shared by the kernels that map gradients of
// rotated rows back to the unrotated rows.
#pragma once
#include <cuda_runtime.h>

namespace nea {

// Rotary embedding, inverse direction, of one pair (a, b) = (x_2i, x_2i+1):
// cs = (cos, sin) of the pair's angle at the row's position.  The forward
// rotation is [[c, -s], [s, c]]; its transpose maps dL/dY to dL/dX.
__device__ __forceinline__ void rope_inv(float& a, float& b, float2 cs) {
  const float x = a, y = b;
  a = fmaf(x, cs.x, y * cs.y);
  b = fmaf(y, cs.x, -(x * cs.y));
}

}  // namespace nea
