// Warp-wide register sorts.
#pragma once

#include "ctcpb_internal.cuh"

namespace ctcpb {

// Bitonic sort, descending, of 32*E keys held E per lane (element i = lane +
// 32*e); one shuffle per element per stage for strides below 32.
template <int E, class T>
__device__ __forceinline__ void warp_sort_desc(T (&v)[E], int lane) {
#pragma unroll
  for (int k = 2; k <= 32 * E; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      if (j >= 32) {
        const int je = j >> 5;
#pragma unroll
        for (int e = 0; e < E; ++e) {
          if ((e & je) == 0) {
            const int i = lane + 32 * e;
            const bool desc = (i & k) == 0;
            const T a = v[e], b = v[e + je];
            const bool sw = desc ? (a < b) : (a > b);
            v[e] = sw ? b : a;
            v[e + je] = sw ? a : b;
          }
        }
      } else {
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const int i = lane + 32 * e;
          const T p = __shfl_xor_sync(0xffffffffu, v[e], j);
          const bool desc = (i & k) == 0, lower = (i & j) == 0;
          const bool keep_max = lower == desc;
          v[e] = keep_max ? (p > v[e] ? p : v[e]) : (p < v[e] ? p : v[e]);
        }
      }
    }
  }
}

}  // namespace ctcpb
