// Host-side entry points of the wide decode kernels (dec_wide.cu).
#pragma once
#include "dec_common.h"

namespace dec {
namespace wide {

using WideKernelFn = void (*)(const KParams, const WideParams);

// the kernel for B operand blocks of nr rows (steps of up to nr / 2 tokens), or null
WideKernelFn kernel_for(int nr, int hd, int group);
// dynamic shared memory of a kernel with `ring` slots
int smem_bytes(int ring, int nr, int hd, int group);
// partial-sum slots per output row block, and tiles, of GEMV stage `kind` with U routed experts
// split over G CTAs
int stage_slots(const KParams& p, int kind, int U, int G);
int stage_tiles(const KParams& p, int kind, int U, int G);

constexpr int kWideTopkHost = 8;  // the wide kernel's experts per token (its routing tables)
constexpr int kWideMinBatch = 5;  // the smallest decode batch the wide kernel takes by default

}  // namespace wide
}  // namespace dec
