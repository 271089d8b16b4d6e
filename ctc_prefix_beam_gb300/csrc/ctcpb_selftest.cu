// Self-test of the decoder's bounded waits: failure detection that needs no
// GPU fault.  The kernels wait in two forms -- an acquire spin over ready
// flags that other blocks set (the fused launch's ranked-record wait) and an
// mbarrier phase (the pre-pass's bulk copies) -- and each wait gives up after
// a bounded number of tries, reporting CTCPB_DEV_TIMEOUT instead of hanging.
// This kernel runs both forms against conditions that never complete: flags
// that nothing sets and a barrier phase that lacks an arrival.
#include "ctcpb_async.cuh"
#include "ctcpb_internal.cuh"

namespace ctcpb {
namespace {

__global__ void __launch_bounds__(32) k_selftest_waits(const u32* __restrict__ flags, int nflags, long long spins,
                                                       u32* __restrict__ out) {
  __shared__ __align__(8) u64 bar;
  const int lane = threadIdx.x;
  // 1. ready flags, acquired up to 32 at a time: lane j tests flag s_pub + j
  int s_pub = 0;
  for (long long spin = 0; s_pub < nflags && spin < spins; ++spin) {
    const int r = s_pub + lane;
    const bool set = r >= nflags || ld_acquire_u32(flags + r) != 0u;
    const unsigned m = __ballot_sync(0xffffffffu, set);
    s_pub += (m == 0xffffffffu) ? 32 : __ffs(~m) - 1;
    if (s_pub < nflags) __nanosleep(64);
  }
  if (s_pub > nflags) s_pub = nflags;
  // 2. a barrier phase that expects two arrivals and receives one
  if (lane == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 2;\n" ::"r"(saddr(&bar)) : "memory");
    mbar_init_fence();
    asm volatile("{\n .reg .b64 st;\n mbarrier.arrive.shared::cta.b64 st, [%0];\n}\n" ::"r"(saddr(&bar)) : "memory");
  }
  __syncwarp();
  const bool phase_done = mbar_wait(&bar, 0u);
  if (lane == 0) {
    out[0] = (u32)s_pub;
    out[1] = s_pub < nflags ? CTCPB_DEV_TIMEOUT : 0u;
    out[2] = phase_done ? 0u : CTCPB_DEV_TIMEOUT;
  }
}

}  // namespace
}  // namespace ctcpb

extern "C" int ctcpb_selftest_waits(const uint32_t* flags, int nflags, long long max_spins, uint32_t* out,
                                    ctcpb_stream_t stream) {
  if (nflags < 0 || max_spins < 1 || max_spins > (1ll << 20)) return CTCPB_EINVAL;
  if (!out || (nflags > 0 && !flags)) return CTCPB_ENULL;
  ctcpb::k_selftest_waits<<<1, 32, 0, (cudaStream_t)stream>>>(flags, nflags, max_spins, out);
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? CTCPB_OK : CTCPB_ECUDA;
}
