// Device primitives of the persistent decode kernel: mbarrier rings fed by bulk (TMA) copies,
// acquire/release flags and counters, and FP8/bf16 conversions. Every wait is
// bounded by %globaltimer: on expiry it records an error code in the device status word and
// returns false, and every caller unwinds without touching the GPU further.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <cstdint>

#include "dec_common.h"

namespace dec {

__device__ __forceinline__ unsigned long long gtimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------------------------------------
// status word

__device__ __forceinline__ bool aborted(const KParams& p) {
  return *reinterpret_cast<volatile int*>(p.err) != 0;
}

static __device__ __noinline__ void raise_err(const KParams& p, int code, int where) {
  atomicCAS(p.err, 0, code | (where << 8));
}


// ---------------------------------------------------------------------------------------------
// mbarrier

__device__ __forceinline__ void mbar_init(uint64_t* b, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(b)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* b, unsigned bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(b)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(b)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_cnt(uint64_t* b, unsigned count) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(b)), "r"(count) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* b, unsigned parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(b)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for phase `parity` of an mbarrier; false on timeout or abort. The first test is inline;
// the polling loop is one out-of-line copy. The clock and the status word (an L2 round trip) are
// consulted only every 64 polls, so a wait that ends quickly costs no global traffic.
static __device__ __noinline__ bool mbar_wait_slow(uint64_t* b, unsigned parity, int* err, unsigned long long timeout_ns,
                                            int where) {
  const unsigned long long t0 = gtimer();
  for (unsigned it = 1;; ++it) {
    if (mbar_try_wait(b, parity)) return true;
    if ((it & 63u) == 0) {
      if (*reinterpret_cast<volatile int*>(err) != 0) return false;
      if (gtimer() - t0 > timeout_ns) {
        atomicCAS(err, 0, kDevTimeout | (where << 8));
        return false;
      }
    }
  }
}
__device__ __forceinline__ bool mbar_wait(uint64_t* b, unsigned parity, const KParams& p, int where) {
  if (mbar_try_wait(b, parity)) return true;
  return mbar_wait_slow(b, parity, p.err, p.timeout_ns, where);
}

// ---------------------------------------------------------------------------------------------
// bulk copies (TMA, non-tensor): global -> this CTA's shared memory, completing on an mbarrier,
// with an L2 eviction-priority hint (a policy made by createpolicy). Addresses 16-byte aligned,
// size a multiple of 16.
__device__ __forceinline__ void bulk_g2s_hint(void* dst, const void* src, unsigned bytes, uint64_t* bar,
                                              uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}
// every access of a copy gets the evict-first priority (its lines leave L2 before others) or
// the normal one
__device__ __forceinline__ uint64_t l2_policy(bool evict_first) {
  uint64_t pol;
  if (evict_first)
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  else
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}


// ---------------------------------------------------------------------------------------------
// cross-CTA memory

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release(unsigned* p, unsigned v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Called by all 32 lanes of one warp: wait until *addr[i] >= want[i] (unsigned, acquire) for
// every i < n with a non-null address; lane j polls conditions j, j + 32, ... Returns 1 when they
// all hold, 0 on abort or after timeout_ns (then the status word records a timeout at `where`).
// One out-of-line copy serves every wait of the kernel.
static __device__ __noinline__ int poll_all_geq(const unsigned* const* addr, const unsigned* want, int n,
                                         int* err, unsigned long long timeout_ns, int where) {
  const int lane = threadIdx.x & 31;
  const unsigned long long t0 = gtimer();
  for (unsigned it = 1;; ++it) {
    bool ok = true;
#pragma unroll 1
    for (int i = lane; i < n; i += 32)
      if (addr[i] && ld_acquire(addr[i]) < want[i]) ok = false;
    if (__all_sync(0xffffffffu, ok)) return 1;
    if ((it & 15u) == 0) {
      int bad = 0;
      if (lane == 0) {
        if (*reinterpret_cast<volatile int*>(err) != 0) bad = 1;
        else if (gtimer() - t0 > timeout_ns) {
          atomicCAS(err, 0, kDevTimeout | (where << 8));
          bad = 1;
        }
      }
      if (__shfl_sync(0xffffffffu, bad, 0)) return 0;
    }
  }
}

// Counter arrival that publishes: the release orders the writes before it (this thread's, and
// through a preceding CTA barrier the whole CTA's) before the increment, without stalling the
// issuing thread the way a full fence does.
__device__ __forceinline__ void red_release_add(int* p, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Arrival without ordering (a count that publishes no data).
__device__ __forceinline__ void red_relaxed_add(int* p, int v) {
  asm volatile("red.relaxed.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ int atom_add_acqrel(int* p, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// L2-coherent loads for data written by other CTAs during this launch (never served from a
// possibly stale L1 line).
__device__ __forceinline__ float ldcg(const float* p) { return __ldcg(p); }
__device__ __forceinline__ uint4 ldcg4(const void* p) { return __ldcg(reinterpret_cast<const uint4*>(p)); }
__device__ __forceinline__ uint16_t ldcg_u16(const uint16_t* p) { return __ldcg(p); }

// Consumer-warp barrier (named barrier 1, 256 threads) that also returns whether v held in any
// of the consumer threads.
__device__ __forceinline__ bool cons_any(bool v) {
  unsigned r;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\tsetp.ne.u32 pi, %1, 0;\n\tbar.red.or.pred po, 1, %2, pi;\n\t"
      "selp.u32 %0, 1, 0, po;\n\t}"
      : "=r"(r)
      : "r"((unsigned)v), "n"(kConsumerWarps * 32)
      : "memory");
  return r != 0;
}

// Consumer warps only (named barrier 1, 256 threads).
__device__ __forceinline__ void cons_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
}


// ---------------------------------------------------------------------------------------------
// 5th-generation tensor cores (tcgen05): tensor memory (TMEM) accumulators, MMAs issued by one
// thread with operands described in shared memory, completion signalled on an mbarrier.

// Allocate ncols TMEM columns (a power of two >= 32) for this CTA; the base address is written to
// *dst (shared). Executed by one whole warp, which must also free them.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)), "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_free(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// Ordering of tensor-core operations across a thread synchronisation (barrier or mbarrier).
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Global memory written through the generic proxy (plain stores, seen through an acquire) made
// visible to this thread's later bulk copies (async proxy).
__device__ __forceinline__ void fence_proxy_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }

// Generic-proxy shared-memory writes (st.shared) made visible to the tensor cores' reads.
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Shared-memory matrix descriptor of an operand without swizzling, made of 128-byte core
// matrices: K-major, 8 rows (M or N) x 16 bytes of K; MN-major, 8 K indices x 16 bytes of M or N.
// lbo: bytes between core matrices adjacent in K; sbo: between those adjacent in M or N.
__device__ __forceinline__ uint64_t smem_desc(const void* base, uint32_t lbo, uint32_t sbo) {
  const uint32_t a = smem_u32(base);
  return (uint64_t)((a & 0x3FFFFu) >> 4) | ((uint64_t)(lbo >> 4) << 16) | ((uint64_t)(sbo >> 4) << 32) |
         (1ull << 46);  // descriptor version 1 (tcgen05); base offset 0; no swizzle
}

// The same for an operand in the 128-byte swizzled layout (atoms of 8 rows x 128 bytes, 1024-byte
// aligned, 16-byte chunks of row r stored at chunk index c ^ (r % 8)). K-major: sbo = bytes between
// 8-row groups (lbo unused); MN-major: lbo = bytes between 64-element atoms along M or N, sbo =
// bytes between groups of 8 K indices.
__device__ __forceinline__ uint64_t smem_desc_sw128(const void* base, uint32_t lbo, uint32_t sbo) {
  return smem_desc(base, lbo, sbo) | (2ull << 61);
}

// 3-D tensor tile load (TMA) global -> this CTA's shared memory, completing on an mbarrier, with an
// L2 eviction-priority hint. The map lives in kernel parameter space; x (the innermost
// coordinate) times the element size must be a multiple of 16 bytes.
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int x, int y, int z, uint64_t* bar,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// Instruction descriptor of kind::f8f6f4 with E4M3 A and B (both K-major) and an fp32 D of
// shape M x N.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int M, int N) {
  return (1u << 4)                          // D format: f32
         | (0u << 7) | (0u << 10)           // A, B format: E4M3
         | ((uint32_t)(N >> 3) << 17)       // N / 8
         | ((uint32_t)(M >> 4) << 24);      // M / 16
}

// D[tmem] (+)= A * B^T for one K = 32 slice of 8-bit operands.
__device__ __forceinline__ void mma_e4m3(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Instruction descriptor of kind::f16 with bf16 A and B and an fp32 D of shape M x N; A either
// K-major or MN-major (a_mn: the M index contiguous in memory), B K-major.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, bool a_mn) {
  return (1u << 4)                          // D format: f32
         | (1u << 7) | (1u << 10)           // A, B format: bf16
         | ((a_mn ? 1u : 0u) << 15)         // A major-ness (1: MN-major)
         | ((uint32_t)(N >> 3) << 17)       // N / 8
         | ((uint32_t)(M >> 4) << 24);      // M / 16
}

// D[tmem] (+)= A * B^T for one K = 16 slice of bf16 operands.
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive (once) on an mbarrier when every tensor-core operation this thread issued so far is done.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// Each thread of a warp reads its TMEM lane (lane quadrant = warp % 4), NC consecutive columns.
template <int NC>
__device__ __forceinline__ void tmem_ld(uint32_t taddr, float (&d)[8]) {
  uint32_t r[8];
  if constexpr (NC == 2) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x2.b32 {%0, %1}, [%2];" : "=r"(r[0]), "=r"(r[1]) : "r"(taddr));
  } else if constexpr (NC == 4) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(taddr));
  } else {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
  }
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 8; ++i) d[i] = i < NC ? __uint_as_float(r[i]) : 0.f;
}

// Wider loads for the wide kernel's epilogue: 16 or 32 consecutive columns of the thread's lane
// (fp32 bit patterns), completed before returning.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&d)[16]) {
  uint32_t r[16];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
               : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) d[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&d)[32]) {
  uint32_t r[32];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
               : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) d[i] = __uint_as_float(r[i]);
}

// TMEM reads of 8 columns for one or two tiles, completed in the same statement (both loads in
// flight before the one wait; the outputs are defined only once they are valid).
__device__ __forceinline__ void tmem_ld8_wait(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_ld8x2_wait(uint32_t ta0, uint32_t ta1, uint32_t (&r)[2][8]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%16];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%8, %9, %10, %11, %12, %13, %14, %15}, [%17];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0][0]), "=r"(r[0][1]), "=r"(r[0][2]), "=r"(r[0][3]), "=r"(r[0][4]), "=r"(r[0][5]), "=r"(r[0][6]),
        "=r"(r[0][7]), "=r"(r[1][0]), "=r"(r[1][1]), "=r"(r[1][2]), "=r"(r[1][3]), "=r"(r[1][4]), "=r"(r[1][5]),
        "=r"(r[1][6]), "=r"(r[1][7])
      : "r"(ta0), "r"(ta1)
      : "memory");
}

// ---------------------------------------------------------------------------------------------
// conversions (CUDA's own FP8 conversion instruction; bf16 -> fp32 is a shift)

__device__ __forceinline__ float2 e4m3x2_to_float2(uint32_t two_codes) {
  __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(two_codes & 0xFFFFu), __NV_E4M3);
  return __half22float2(*reinterpret_cast<const __half2*>(&h));
}

// two E4M3 codes (low 16 bits) -> packed f16x2, exact (every E4M3 value is an f16 value)
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_codes) {
  __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(two_codes & 0xFFFFu), __NV_E4M3);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// acc0 += lo(w) * lo(x), acc1 += hi(w) * hi(x): f16 operands, fp32 product-and-sum (one rounding)
__device__ __forceinline__ void fma_f16x2_f32(uint32_t w2, uint32_t x2, float& acc0, float& acc1) {
  asm("{\n\t.reg .f16 wl, wh, xl, xh;\n\t"
      "mov.b32 {wl, wh}, %2;\n\t"
      "mov.b32 {xl, xh}, %3;\n\t"
      "fma.rn.f32.f16 %0, wl, xl, %0;\n\t"
      "fma.rn.f32.f16 %1, wh, xh, %1;\n\t}"
      : "+f"(acc0), "+f"(acc1)
      : "r"(w2), "r"(x2));
}

// two floats -> two E4M3 codes (round to nearest even, saturating to +-448), low code first
__device__ __forceinline__ uint16_t float2_to_e4m3x2(float lo, float hi) {
  return static_cast<uint16_t>(__nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3));
}

__device__ __forceinline__ float bf16lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }
__device__ __forceinline__ float bf16f(uint16_t u) { return __uint_as_float(static_cast<uint32_t>(u) << 16); }

__device__ __forceinline__ uint16_t f2bf(float f) {
  __nv_bfloat16 b = __float2bfloat16_rn(f);
  return *reinterpret_cast<uint16_t*>(&b);
}

// Order-preserving map float -> uint32 (larger float -> larger key).
__device__ __forceinline__ uint32_t float_key(float f) {
  uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

}  // namespace dec
