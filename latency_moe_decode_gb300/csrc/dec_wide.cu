// The wide decode kernels (steps of 5 .. 64 tokens), compiled in their own translation unit.
#include "dec_wide.cuh"
#include "dec_wide_host.h"

namespace dec {
namespace wide {

WideKernelFn kernel_for(int nr, int hd, int group) {
#define DEC_WK(N, H, GR) \
  if (nr == N && hd == H && group == GR) return wide_step_kernel<N, H, GR>;
  DEC_WK(32, 64, 2) DEC_WK(64, 64, 2) DEC_WK(128, 64, 2)
  DEC_WK(32, 128, 4) DEC_WK(64, 128, 4) DEC_WK(128, 128, 4)
#undef DEC_WK
  return nullptr;
}

int smem_bytes(int ring, int nr, int hd, int group) { return wlayout(ring, nr, hd, group).total; }

int stage_slots(const KParams& p, int kind, int U, int G) { return wgeo(p, kind, U, G).S; }
int stage_tiles(const KParams& p, int kind, int U, int G) { return wgeo(p, kind, U, G).T; }

}  // namespace wide
}  // namespace dec
