// The persistent decode-step kernel.
//
// One launch runs a whole decode step: for every layer, RMSNorm + q/k/v projection + RoPE + KV
// append, split-KV GQA attention with an in-kernel merge, output projection + residual,
// RMSNorm + sigmoid router + top-k, the shared expert, the routed SwiGLU experts, the
// gate-weighted combine + residual; then the final RMSNorm, the LM head and the greedy argmax.
// ("Ultra-High Interactivity on NVIDIA GPUs? TileRT on InferenceX", section "But What Exactly is
// TileRT?": one resident kernel instead of a kernel per operator, warp groups specialised on
// data movement and compute, tile-granular overlap, intermediates kept on chip / in L2. The
// per-layer recipe follows "vLLM's Kimi K3 Backend Hits 842 Tokens per Second", section "Four
// changes drive the gains".)
//
// Structure of a CTA (one per SM, all co-resident):
//   warp 8      producer: walks the CTA's static load program and streams weight tiles (and KV
//               tiles) into a ring of shared-memory slots with 1-D bulk copies (TMA) completing
//               on mbarriers. Static weights never depend on activations, so the producer runs
//               ahead across stage boundaries (the fix named on the vLLM page, section "Agent-
//               written kernels face evidence gates": only static weights are loaded ahead of a
//               synchronisation wait). While the routed experts are unknown it issues L2
//               prefetches of its next-layer tiles, so HBM stays busy through the routing bubble.
//   warps 0..7  consumers: dequantise E4M3 tiles (CUDA's cvt), multiply by the bf16 activations
//               held in shared memory, accumulate in fp32, reduce across warps, and publish
//               split-K partial sums. The last CTA to publish a partial of an output block
//               finalises it (RoPE/KV append, residual add, SwiGLU, routing, logits + argmax):
//               the "last arriver" pattern replaces a second pass.
// Stage boundaries are grid-wide barriers on a generation counter (acquire/release); there are
// five per layer. Every wait is bounded and turns into an error status instead of a hang.
#pragma once
#include "dec_prims.cuh"

namespace dec {

// ---------------------------------------------------------------------------------------------
// shared-memory layout (identical on host and device)

struct SmemLayout {
  int ring_off, full_off, empty_off, xs_off, red_off, misc_off, total;
};

constexpr int kMaxExperts = 128;

struct Misc {
  int flag;
  int nfin;
  int U;
  int v_lo;
  int len[kMaxBatch];
  int fin_group[64];
  int fin_old[64];
  int elist[kMaxExperts];
  float gate[kMaxBatch][kMaxExperts + 1];
  float rsum[kConsumerWarps][kMaxBatch];
  int tok[kMaxBatch];
};

__host__ __device__ inline int align_up(int x, int a) { return (x + a - 1) / a * a; }

__host__ __device__ inline SmemLayout smem_layout(int ring, int bm, int xmax, int hd, int group) {
  SmemLayout s;
  s.ring_off = 0;
  s.full_off = align_up(ring * kSlotBytes, 128);
  s.empty_off = s.full_off + ring * 8;
  s.xs_off = align_up(s.empty_off + ring * 8, 128);
  s.red_off = align_up(s.xs_off + bm * xmax * 2, 128);
  int red_gemv = kConsumerWarps * kTileRows * bm * 4;
  int red_attn = kConsumerWarps * group * (hd + 2) * 4;
  int red = red_gemv > red_attn ? red_gemv : red_attn;
  s.misc_off = align_up(s.red_off + red, 128);
  s.total = align_up(s.misc_off + (int)sizeof(Misc), 128);
  return s;
}

// GEMV stage kinds
enum Kind : int { K_QKV = 0, K_O, K_ROUTER, K_SHGU, K_RTGU, K_D, K_LM };

// ---------------------------------------------------------------------------------------------
// schedule arithmetic shared by producer and consumers

__device__ __forceinline__ int range_lo(int T, int c, int G) { return (int)((long long)T * c / G); }
__device__ __forceinline__ int owner_of(int t, int T, int G) {
  return (int)(((long long)(t + 1) * G - 1) / T);
}
// contributors to a segment of kbs consecutive tiles starting at tile a
__device__ __forceinline__ int n_contrib(int a, int kbs, int T, int G) {
  if (T < G) return kbs;
  return owner_of(a + kbs - 1, T, G) - owner_of(a, T, G) + 1;
}
// slot of CTA c (whose first tile inside the segment is f) among the segment's contributors
__device__ __forceinline__ int contrib_slot(int c, int f, int a, int T, int G) {
  if (T < G) return f - a;
  return c - owner_of(a, T, G);
}

struct StageGeo {
  int T;    // tiles
  int kbs;  // tiles per segment
  int tpe;  // tiles per expert (routed / down stages)
};

__device__ __forceinline__ StageGeo stage_geo(const KParams& p, int kind, int U) {
  StageGeo g;
  g.tpe = 0;
  switch (kind) {
    case K_QKV: g.kbs = p.kb_d; g.T = p.n_rb_qkv * p.kb_d; break;
    case K_O: g.kbs = p.kb_o; g.T = p.n_rb_d * p.kb_o; break;
    case K_ROUTER: g.kbs = p.kb_d; g.T = p.n_rb_router * p.kb_d; break;
    case K_SHGU: g.kbs = p.kb_d; g.T = p.n_rb_gu * p.kb_d; break;
    case K_RTGU: g.kbs = p.kb_d; g.tpe = p.n_rb_gu * p.kb_d; g.T = U * g.tpe; break;
    case K_D: g.kbs = p.kb_i; g.tpe = p.n_rb_d * p.kb_i; g.T = (U + p.nsh) * g.tpe; break;
    default: g.kbs = p.kb_d; g.T = p.n_rb_lm * p.kb_d; break;
  }
  return g;
}

__device__ __forceinline__ const uint8_t* tile_addr(const KParams& p, const LayerDev& Ld, int kind,
                                                    int t, const StageGeo& g, int U, const int* elist) {
  const size_t TB = kTileBytes;
  switch (kind) {
    case K_QKV: return Ld.qkv + (size_t)t * TB;
    case K_O: return Ld.o + (size_t)t * TB;
    case K_ROUTER: return Ld.router + (size_t)t * TB;
    case K_SHGU: return Ld.sh_gu + (size_t)t * TB;
    case K_RTGU: {
      int u = t / g.tpe, r = t - u * g.tpe;
      return Ld.e_gu + (size_t)elist[u] * p.e_gu_stride + (size_t)r * TB;
    }
    case K_D: {
      int v = t / g.tpe, r = t - v * g.tpe;
      if (v < U) return Ld.e_d + (size_t)elist[v] * p.e_d_stride + (size_t)r * TB;
      return Ld.sh_d + (size_t)r * TB;
    }
    default: return p.lm + (size_t)t * TB;
  }
}

// attention work units: (sequence b, KV head g, context chunk c)
struct AttnUnit {
  int b, g, c, tile0, tile1, T;
};
__device__ __forceinline__ AttnUnit attn_unit(const KParams& p, const Misc* m, int u) {
  AttnUnit a;
  int per_b = p.hkv * p.nch;
  a.b = u / per_b;
  a.g = (u / p.nch) % p.hkv;
  a.c = u % p.nch;
  a.T = m->len[a.b] + 1;
  int ntile = (a.T + kKvTilePos - 1) / kKvTilePos;
  int tpc = (ntile + p.nch - 1) / p.nch;
  a.tile0 = min(ntile, a.c * tpc);
  a.tile1 = min(ntile, a.tile0 + tpc);
  return a;
}

__device__ __forceinline__ size_t kv_row(const KParams& p, int l, int b, int g, int pos) {
  return ((((size_t)l * p.MB + (p.seq0 + b)) * p.hkv + g) * p.max_ctx + pos) * p.hd;
}

// ---------------------------------------------------------------------------------------------
// producer warp

template <int BM, int HD, int G>
struct Producer {
  const KParams& p;
  uint8_t* ring;
  uint64_t* full;
  uint64_t* empty;
  Misc* m;
  unsigned item = 0;
  bool dead = false;

  __device__ Producer(const KParams& p_, uint8_t* r, uint64_t* f, uint64_t* e, Misc* m_)
      : p(p_), ring(r), full(f), empty(e), m(m_) {}

  // claim the next slot: wait until the consumers released it
  __device__ bool claim(int& slot) {
    slot = item % p.ring;
    if (item >= (unsigned)p.ring) {
      unsigned par = ((item / p.ring) - 1) & 1;
      if (!mbar_wait(&empty[slot], par, p, 10)) {
        dead = true;
        return false;
      }
    }
    return true;
  }

  __device__ void issue_gemv(int kind, int l, int U, const int* elist) {
    if (dead) return;
    const StageGeo g = stage_geo(p, kind, U);
    const int G_ = gridDim.x;
    const int t0 = range_lo(g.T, blockIdx.x, G_), t1 = range_lo(g.T, blockIdx.x + 1, G_);
    const LayerDev& Ld = p.layers[l < p.L ? l : 0];
    for (int t = t0; t < t1; ++t) {
      int slot;
      if (!claim(slot)) return;
      const uint8_t* src = tile_addr(p, Ld, kind, t, g, U, elist);
      uint8_t* dst = ring + (size_t)slot * kSlotBytes;
      mbar_arrive_expect_tx(&full[slot], kTileBytes);
      bulk_g2s(dst, src, kTileBytes, &full[slot]);
      ++item;
    }
  }

  __device__ void prefetch_gemv(int kind, int l) {
    if (dead) return;
    const StageGeo g = stage_geo(p, kind, 0);
    const int t0 = range_lo(g.T, blockIdx.x, gridDim.x), t1 = range_lo(g.T, blockIdx.x + 1, gridDim.x);
    const LayerDev& Ld = p.layers[l < p.L ? l : 0];
    const int tmax = t0 + 24;  // at most ~390 KB per stage and CTA
    for (int t = t0; t < t1 && t < tmax; ++t) prefetch_l2(tile_addr(p, Ld, kind, t, g, 0, nullptr), kTileBytes);
  }

  __device__ void issue_attn(int l) {
    if (dead) return;
    const int NU = p.B * p.hkv * p.nch;
    const unsigned row_bytes = HD * 2;
    for (int u = blockIdx.x; u < NU; u += gridDim.x) {
      AttnUnit a = attn_unit(p, m, u);
      for (int t = a.tile0; t < a.tile1; ++t) {
        int slot;
        if (!claim(slot)) return;
        int p0 = t * kKvTilePos;
        int n = min(kKvTilePos, a.T - p0);
        uint8_t* dst = ring + (size_t)slot * kSlotBytes;
        const size_t r0 = kv_row(p, l, a.b, a.g, p0);
        mbar_arrive_expect_tx(&full[slot], 2u * n * row_bytes);
        bulk_g2s(dst, p.kc + r0, n * row_bytes, &full[slot]);
        bulk_g2s(dst + kKvTilePos * row_bytes, p.vc + r0, n * row_bytes, &full[slot]);
        ++item;
      }
    }
  }

  __device__ void prefetch_attn(int l) {
    if (dead) return;
    const int NU = p.B * p.hkv * p.nch;
    for (int u = blockIdx.x; u < NU; u += gridDim.x) {
      AttnUnit a = attn_unit(p, m, u);
      if (a.tile1 <= a.tile0) continue;
      int n = min(a.T, a.tile1 * kKvTilePos) - a.tile0 * kKvTilePos;
      const size_t r0 = kv_row(p, l, a.b, a.g, a.tile0 * kKvTilePos);
      prefetch_l2(p.kc + r0, (unsigned)n * HD * 2);
      prefetch_l2(p.vc + r0, (unsigned)n * HD * 2);
    }
  }

  // Routed experts are known only after the router: wait for this layer's routing flag.
  __device__ bool routing(int l, int& U, int* elist) {
    if (dead) return false;
    if (!wait_flag(p, p.rt_flag + l, p.epoch, 11)) {
      dead = true;
      return false;
    }
    U = min(max(__ldcg(p.rt_u), 0), p.umax);
    for (int i = 0; i < U; ++i) elist[i] = min(max(__ldcg(p.rt_elist + i), 0), p.E - 1);
    return true;
  }

  // after an abort: let every copy already issued land before the CTA may exit
  __device__ void drain() {
    unsigned first = item > (unsigned)p.ring ? item - p.ring : 0u;
    for (unsigned i = first; i < item; ++i) {
      int slot = i % p.ring;
      unsigned par = (i / p.ring) & 1;
      const unsigned long long t0 = gtimer();
      while (!mbar_try_wait(&full[slot], par)) {
        if (gtimer() - t0 > p.timeout_ns) break;
      }
    }
  }

  __device__ void run() {
    int elist[kMaxExperts];
    for (int l = 0; l < p.L; ++l) {
      issue_gemv(K_QKV, l, 0, nullptr);
      issue_attn(l);
      issue_gemv(K_O, l, 0, nullptr);
      if (p.dense) {
        issue_gemv(K_SHGU, l, 0, nullptr);
        issue_gemv(K_D, l, 0, nullptr);
      } else {
        issue_gemv(K_ROUTER, l, 0, nullptr);
        if (p.nsh) issue_gemv(K_SHGU, l, 0, nullptr);
        // fill the routing bubble with L2 prefetches of what this CTA loads next
        if (l + 1 < p.L) {
          prefetch_gemv(K_QKV, l + 1);
          prefetch_attn(l + 1);
          prefetch_gemv(K_O, l + 1);
        } else if (p.V > 0) {
          prefetch_gemv(K_LM, 0);
        }
        int U = 0;
        if (!routing(l, U, elist)) break;
        issue_gemv(K_RTGU, l, U, elist);
        issue_gemv(K_D, l, U, elist);
      }
      if (dead) break;
    }
    if (!dead && p.V > 0) issue_gemv(K_LM, 0, 0, nullptr);
    if (dead) drain();
  }
};

// ---------------------------------------------------------------------------------------------
// consumer warps

template <int BM, int HD, int G>
struct Consumer {
  const KParams& p;
  uint8_t* ring;
  uint64_t* full;
  uint64_t* empty;
  uint16_t* xs;
  float* red;
  Misc* m;
  unsigned item = 0;
  bool dead = false;
  int warp, lane, tid;
  int stamp = 0;

  __device__ Consumer(const KParams& p_, uint8_t* r, uint64_t* f, uint64_t* e, uint16_t* x, float* rd,
                      Misc* m_)
      : p(p_), ring(r), full(f), empty(e), xs(x), red(rd), m(m_) {
    tid = threadIdx.x;
    warp = tid >> 5;
    lane = tid & 31;
  }

  __device__ void trace() {
    if (blockIdx.x == 0 && tid == 0 && stamp < kTraceSlots) p.trace[stamp++] = gtimer();
  }

  __device__ bool gsync(int where) {
    if (dead) {
      // keep the named-barrier sequence identical across warps; no grid traffic
      cons_sync();
      cons_sync();
      return false;
    }
    bool ok = grid_sync(p, &m->flag, where);
    if (!ok) dead = true;
    trace();
    return ok;
  }

  __device__ const uint8_t* wait_item() {
    int slot = item % p.ring;
    if (!dead) {
      if (!mbar_wait(&full[slot], (item / p.ring) & 1, p, 20)) dead = true;
    }
    return ring + (size_t)slot * kSlotBytes;
  }
  __device__ void release_item() {
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[item % p.ring]);
    ++item;
  }

  // -------- activation staging --------

  __device__ const uint16_t* x_in(int l, int b) const {
    if (l > 0) return p.xbuf + ((size_t)(l & 1) * p.MB + b) * p.d;
    if (p.tokens) return p.embed + (size_t)m->tok[b] * p.d;
    return p.hidden_in + (size_t)b * p.d;
  }

  // xs[b][0..d) = bf16(rmsnorm(src_b) * w); one pass for the sum of squares, one to write.
  __device__ void stage_rmsnorm(int l_src, const uint16_t* direct, const uint16_t* w) {
    for (int b = 0; b < p.B; ++b) {
      const uint16_t* src = direct ? direct + (size_t)b * p.d : x_in(l_src, b);
      float ss = 0.f;
      for (int k = tid * 8; k < p.d; k += kConsumerWarps * 32 * 8) {
        uint4 v = ldcg4(src + k);
        const uint32_t* u = reinterpret_cast<const uint32_t*>(&v);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          float a = bf16lo(u[j]), c = bf16hi(u[j]);
          ss = fmaf(a, a, ss);
          ss = fmaf(c, c, ss);
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      if (lane == 0) m->rsum[warp][b] = ss;
    }
    cons_sync();
    for (int b = 0; b < p.B; ++b) {
      float ss = 0.f;
#pragma unroll
      for (int wi = 0; wi < kConsumerWarps; ++wi) ss += m->rsum[wi][b];
      const float inv = 1.0f / sqrtf(ss / (float)p.d + p.eps);
      const uint16_t* src = direct ? direct + (size_t)b * p.d : x_in(l_src, b);
      for (int k = tid * 8; k < p.d; k += kConsumerWarps * 32 * 8) {
        uint4 v = ldcg4(src + k);
        uint4 wv = *reinterpret_cast<const uint4*>(w + k);
        const uint32_t* u = reinterpret_cast<const uint32_t*>(&v);
        const uint32_t* wu = reinterpret_cast<const uint32_t*>(&wv);
        uint4 o;
        uint32_t* ou = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint16_t lo = f2bf((bf16lo(u[j]) * inv) * bf16lo(wu[j]));
          uint16_t hi = f2bf((bf16hi(u[j]) * inv) * bf16hi(wu[j]));
          ou[j] = (uint32_t)lo | ((uint32_t)hi << 16);
        }
        *reinterpret_cast<uint4*>(xs + (size_t)b * p.xmax + k) = o;
      }
    }
    cons_sync();
  }

  // xs[b][0..n) = src[b][0..n) for a bf16 activation written by other CTAs
  __device__ void stage_copy(const uint16_t* src, int n, size_t src_stride, int dst_off) {
    for (int b = 0; b < p.B; ++b)
      for (int k = tid * 8; k < n; k += kConsumerWarps * 32 * 8)
        *reinterpret_cast<uint4*>(xs + (size_t)b * p.xmax + dst_off + k) = ldcg4(src + (size_t)b * src_stride + k);
  }

  // -------- split-K GEMV over one stage --------

  __device__ __forceinline__ void tile_dot(const uint8_t* tile, int xoff, const float* gmul,
                                           float (&acc)[4][BM]) {
    uint4 wv[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      wv[i] = *reinterpret_cast<const uint4*>(tile + (((i * kConsumerWarps + warp) * 32 + lane) << 4));
    const float2 sc = *reinterpret_cast<const float2*>(tile + kTileData);
    float wf[4][16];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t* u = reinterpret_cast<const uint32_t*>(&wv[i]);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        float2 a = e4m3x2_to_float2(u[j]);
        float2 c = e4m3x2_to_float2(u[j] >> 16);
        wf[i][4 * j + 0] = a.x;
        wf[i][4 * j + 1] = a.y;
        wf[i][4 * j + 2] = c.x;
        wf[i][4 * j + 3] = c.y;
      }
    }
#pragma unroll
    for (int b = 0; b < BM; ++b) {
      if (b < p.B) {
        const uint16_t* xp = xs + (size_t)b * p.xmax + xoff + warp * 16;
        uint4 x0 = *reinterpret_cast<const uint4*>(xp);
        uint4 x1 = *reinterpret_cast<const uint4*>(xp + 8);
        const uint32_t* xu0 = reinterpret_cast<const uint32_t*>(&x0);
        const uint32_t* xu1 = reinterpret_cast<const uint32_t*>(&x1);
        float2 xf[8];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          xf[j] = make_float2(bf16lo(xu0[j]), bf16hi(xu0[j]));
          xf[4 + j] = make_float2(bf16lo(xu1[j]), bf16hi(xu1[j]));
        }
        const float g = gmul[b];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          float2 s2 = make_float2(0.f, 0.f);
#pragma unroll
          for (int j = 0; j < 8; ++j) s2 = __ffma2_rn(make_float2(wf[i][2 * j], wf[i][2 * j + 1]), xf[j], s2);
          const float sc_i = (i < 2 ? sc.x : sc.y) * g;
          acc[i][b] = fmaf(sc_i, s2.x + s2.y, acc[i][b]);
        }
      }
    }
  }

  __device__ float* part_base(int kind) const {
    switch (kind) {
      case K_QKV: return p.part_qkv;
      case K_O: return p.part_o;
      case K_ROUTER: return p.part_router;
      case K_SHGU: return p.part_shgu;
      case K_RTGU: return p.part_rtgu;
      case K_D: return p.part_d;
      default: return p.part_lm;
    }
  }
  __device__ int* cnt_base(int kind) const {
    switch (kind) {
      case K_QKV: return p.cnt_qkv;
      case K_O: return p.cnt_o;
      case K_ROUTER: return p.cnt_router;
      case K_SHGU: return p.cnt_shgu;
      case K_RTGU: return p.cnt_rtgu;
      case K_D: return p.cnt_d;
      default: return p.cnt_lm;
    }
  }
  // output group of a segment (D: the output row block shared by all experts)
  __device__ __forceinline__ int seg_group(int kind, int seg) const {
    return kind == K_D ? seg % p.n_rb_d : seg;
  }

  // Cross-warp reduction of one segment's accumulators, publication of the CTA's partial sums,
  // and the arrival on the output group's counter (result kept for the end of the stage).
  __device__ void flush(int kind, const StageGeo& g, int seg, int first_tile, float (&acc)[4][BM]) {
    // red[w][row][b]
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int b = 0; b < BM; ++b) red[((size_t)warp * kTileRows + i * 32 + lane) * BM + b] = acc[i][b];
    cons_sync();
    const int a = seg * g.kbs;
    const int slot = contrib_slot(blockIdx.x, first_tile, a, g.T, gridDim.x);
    float* dst = part_base(kind) + ((size_t)seg * g.kbs + slot) * p.MB * kTileRows;
    for (int idx = tid; idx < p.B * kTileRows; idx += kConsumerWarps * 32) {
      const int b = idx / kTileRows, row = idx % kTileRows;
      float s = 0.f;
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) s += red[((size_t)w * kTileRows + row) * BM + b];
      dst[(size_t)b * kTileRows + row] = s;
    }
    __threadfence();
    cons_sync();
    if (tid == 0) {
      const int grp = seg_group(kind, seg);
      const int n = m->nfin;
      if (n < 64) {
        m->fin_group[n] = grp;
        m->fin_old[n] = dead ? -1 : atom_add_acqrel(cnt_base(kind) + grp, 1);
        m->nfin = n + 1;
      }
    }
  }

  // number of arrivals that complete an output group
  __device__ int group_expected(int kind, const StageGeo& g, int grp) const {
    if (kind != K_D) return n_contrib(grp * g.kbs, g.kbs, g.T, gridDim.x);
    int tot = 0;
    const int nv = g.T / g.tpe;
    for (int v = 0; v < nv; ++v) {
      int seg = v * p.n_rb_d + grp;
      tot += n_contrib(seg * g.kbs, g.kbs, g.T, gridDim.x);
    }
    return tot;
  }

  // sum of the published partials of segment seg for (b, row)
  __device__ __forceinline__ float seg_sum(int kind, const StageGeo& g, int seg, int b, int row) const {
    const int nc = n_contrib(seg * g.kbs, g.kbs, g.T, gridDim.x);
    const float* src = part_base(kind) + (size_t)seg * g.kbs * p.MB * kTileRows + (size_t)b * kTileRows + row;
    float s = 0.f;
    for (int c = 0; c < nc; ++c) s += ldcg(src + (size_t)c * p.MB * kTileRows);
    return s;
  }

  __device__ void gemv_stage(int kind, int l, int U) {
    const StageGeo g = stage_geo(p, kind, U);
    const int G_ = gridDim.x;
    const int t0 = range_lo(g.T, blockIdx.x, G_), t1 = range_lo(g.T, blockIdx.x + 1, G_);
    if (tid == 0) m->nfin = 0;
    cons_sync();
    float gmul[BM];
    float acc[4][BM];
    int seg_cur = -1, seg_first = 0;
    for (int t = t0; t < t1; ++t) {
      const int seg = t / g.kbs;
      if (seg != seg_cur) {
        if (seg_cur >= 0) flush(kind, g, seg_cur, seg_first, acc);
        seg_cur = seg;
        seg_first = t;
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int b = 0; b < BM; ++b) acc[i][b] = 0.f;
      }
      int xoff = (t % g.kbs) * kTileK;
#pragma unroll
      for (int b = 0; b < BM; ++b) gmul[b] = 1.f;
      if (kind == K_D) {
        const int v = t / g.tpe;
        xoff += (v - m->v_lo) * p.inter;
#pragma unroll
        for (int b = 0; b < BM; ++b) gmul[b] = m->gate[b][min(v, kMaxExperts)];
      }
      const uint8_t* tile = wait_item();
      if (!dead) tile_dot(tile, xoff, gmul, acc);
      release_item();
    }
    if (seg_cur >= 0) flush(kind, g, seg_cur, seg_first, acc);
    cons_sync();
    // finalise the output groups this CTA completed
    const int nf = m->nfin;
    for (int f = 0; f < nf; ++f) {
      const int grp = m->fin_group[f];
      const int old = m->fin_old[f];
      if (old < 0 || old + 1 != group_expected(kind, g, grp)) continue;
      __threadfence();
      finalize(kind, l, g, grp, U);
      cons_sync();
      if (tid == 0) atomicExch(cnt_base(kind) + grp, 0);
    }
  }

  // -------- finalisers (run by the CTA whose arrival completed an output group) --------

  __device__ void finalize(int kind, int l, const StageGeo& g, int grp, int U) {
    float* tmp = red;  // [BM][128]
    switch (kind) {
      case K_QKV: {
        for (int idx = tid; idx < p.B * kTileRows; idx += 256) {
          int b = idx / kTileRows, i = idx % kTileRows;
          tmp[b * kTileRows + i] = seg_sum(kind, g, grp, b, i);
        }
        cons_sync();
        const int hq_rows = p.hq * HD, hk_rows = p.hkv * HD;
        for (int idx = tid; idx < p.B * kTileRows; idx += 256) {
          int b = idx / kTileRows, i = idx % kTileRows;
          int r = grp * kTileRows + i;
          if (r >= hq_rows + 2 * hk_rows) continue;
          float val = tmp[b * kTileRows + i];
          int ih = r % HD;
          const int pos = m->len[b];
          if (r < hq_rows + hk_rows) {  // q or k: rotate the (ih, ih + HD/2) pair
            int j = ih % (HD / 2);
            float2 cs = p.rope[(size_t)pos * (HD / 2) + j];
            int partner = (ih < HD / 2) ? i + HD / 2 : i - HD / 2;
            float other = tmp[b * kTileRows + partner];
            val = (ih < HD / 2) ? val * cs.x - other * cs.y : val * cs.x + other * cs.y;
          }
          uint16_t bv = f2bf(val);
          if (r < hq_rows) {
            p.qbuf[(size_t)b * hq_rows + r] = bv;
          } else if (r < hq_rows + hk_rows) {
            int gh = (r - hq_rows) / HD;
            p.kc[kv_row(p, l, b, gh, pos) + ih] = bv;
          } else {
            int gh = (r - hq_rows - hk_rows) / HD;
            p.vc[kv_row(p, l, b, gh, pos) + ih] = bv;
          }
        }
        break;
      }
      case K_O: {
        for (int idx = tid; idx < p.B * kTileRows; idx += 256) {
          int b = idx / kTileRows, i = idx % kTileRows;
          int r = grp * kTileRows + i;
          float y = seg_sum(kind, g, grp, b, i);
          float x = bf16f(ldcg_u16(x_in(l, b) + r));
          p.xmid[(size_t)b * p.d + r] = f2bf(x + y);
        }
        break;
      }
      case K_ROUTER: {
        for (int idx = tid; idx < p.B * kTileRows; idx += 256) {
          int b = idx / kTileRows, i = idx % kTileRows;
          tmp[b * kTileRows + i] = (i < p.E) ? seg_sum(kind, g, grp, b, i) : -INFINITY;
        }
        cons_sync();
        int* mark = reinterpret_cast<int*>(tmp + BM * kTileRows);  // [128]
        if (tid < kMaxExperts) mark[tid] = 0;
        cons_sync();
        if (tid < p.B) {
          const int b = tid;
          const float* r = tmp + b * kTileRows;
          unsigned long long taken0 = 0, taken1 = 0;
          int sel[16];
          float sc[16];
          float sum = 0.f;
          for (int j = 0; j < p.topk; ++j) {
            int best = -1;
            for (int e = 0; e < p.E; ++e) {
              bool tk = e < 64 ? ((taken0 >> e) & 1ull) : ((taken1 >> (e - 64)) & 1ull);
              if (!tk && (best < 0 || r[e] > r[best])) best = e;
            }
            if (best < 64) taken0 |= 1ull << best; else taken1 |= 1ull << (best - 64);
            sel[j] = best;
            sc[j] = 1.0f / (1.0f + expf(-r[best]));
            sum += sc[j];
          }
          for (int j = 0; j < p.topk; ++j) {
            atomicOr(&mark[sel[j]], 1);
            p.rt_idx[((size_t)l * p.MB + b) * p.topk + j] = sel[j];
            p.rt_topk_gate[((size_t)l * p.MB + b) * p.topk + j] = sc[j] / sum;
          }
        }
        cons_sync();
        if (tid == 0) {
          int U2 = 0;
          for (int e = 0; e < p.E; ++e)
            if (mark[e]) {
              mark[e] = U2 + 1;  // 1-based rank of expert e in the distinct list
              p.rt_elist[U2++] = e;
            }
          p.rt_u[0] = U2;
        }
        cons_sync();
        for (int idx = tid; idx < p.B * p.E; idx += 256) {
          int b = idx / p.E, e = idx % p.E;
          if (mark[e] == 0) continue;
          float gt = 0.f;
          for (int j = 0; j < p.topk; ++j)
            if (p.rt_idx[((size_t)l * p.MB + b) * p.topk + j] == e)
              gt = p.rt_topk_gate[((size_t)l * p.MB + b) * p.topk + j];
          p.rt_gate[(size_t)b * kMaxExperts + (mark[e] - 1)] = gt;
        }
        __threadfence();
        cons_sync();
        if (tid == 0) st_release(p.rt_flag + l, p.epoch);
        break;
      }
      case K_SHGU:
      case K_RTGU: {
        const int half = kTileRows / 2;
        int seg = grp;
        int u = 0, rb = grp;
        if (kind == K_RTGU) {
          u = grp / p.n_rb_gu;
          rb = grp % p.n_rb_gu;
        }
        for (int idx = tid; idx < p.B * half; idx += 256) {
          int b = idx / half, i = idx % half;
          float gv = seg_sum(kind, g, seg, b, i);
          float uv = seg_sum(kind, g, seg, b, i + half);
          float h = (gv / (1.0f + expf(-gv))) * uv;
          int j = rb * half + i;
          if (kind == K_SHGU)
            p.hsh[(size_t)b * p.inter + j] = f2bf(h);
          else
            p.hrt[((size_t)u * p.MB + b) * p.inter + j] = f2bf(h);
        }
        break;
      }
      case K_D: {
        const int nv = g.T / g.tpe;
        for (int idx = tid; idx < p.B * kTileRows; idx += 256) {
          int b = idx / kTileRows, i = idx % kTileRows;
          int r = grp * kTileRows + i;
          float y = 0.f;
          for (int v = 0; v < nv; ++v) y += seg_sum(kind, g, v * p.n_rb_d + grp, b, i);
          float x = bf16f(ldcg_u16(p.xmid + (size_t)b * p.d + r));
          uint16_t o = f2bf(x + y);
          p.xbuf[((size_t)((l + 1) & 1) * p.MB + b) * p.d + r] = o;
          if (l == p.L - 1 && p.hidden_out) p.hidden_out[(size_t)b * p.d + r] = o;
        }
        break;
      }
      default: {  // LM head
        float* out = p.logits ? p.logits : p.logits_ws;
        for (int idx = tid; idx < p.B * kTileRows; idx += 256) {
          int b = idx / kTileRows, i = idx % kTileRows;
          int r = grp * kTileRows + i;
          float v = -INFINITY;
          if (r < p.V) {
            v = seg_sum(kind, g, grp, b, i);
            out[(size_t)b * p.V + r] = v;
          }
          tmp[b * kTileRows + i] = v;
        }
        cons_sync();
        if (tid < p.B) {
          const int b = tid;
          int best = 0;
          for (int i = 1; i < kTileRows; ++i)
            if (tmp[b * kTileRows + i] > tmp[b * kTileRows + best]) best = i;
          unsigned long long key = ((unsigned long long)float_key(tmp[b * kTileRows + best]) << 32) |
                                   (unsigned long long)(0xFFFFFFFFu - (unsigned)(grp * kTileRows + best));
          atomicMax(p.amax + b, key);
        }
        __threadfence();
        cons_sync();
        if (tid == 0) {
          int old = atom_add_acqrel(p.cnt_lm_done, 1);
          if (old + 1 == p.n_rb_lm) {
            __threadfence();
            for (int b = 0; b < p.B; ++b) {
              unsigned long long key = atomicExch(p.amax + b, 0ull);
              if (p.next_tokens) p.next_tokens[b] = (int)(0xFFFFFFFFu - (unsigned)(key & 0xFFFFFFFFull));
            }
            atomicExch(p.cnt_lm_done, 0);
          }
        }
        break;
      }
    }
  }

  // -------- split-KV GQA attention --------

  // Reduce NV partial values across the warp; afterwards lane l holds the total of value
  // index l / (32 / NV).
  template <int NV>
  __device__ __forceinline__ float warp_transpose_reduce(float (&v)[NV]) {
#pragma unroll
    for (int off = 16, n = NV; n > 1; off >>= 1, n >>= 1) {
      const bool upper = (lane & off) != 0;
#pragma unroll
      for (int i = 0; i < n / 2; ++i) {
        float send = upper ? v[i] : v[i + n / 2];
        float keep = upper ? v[i + n / 2] : v[i];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
      }
    }
    float r = v[0];
    // remaining butterfly levels sum the lanes that share a value index
    constexpr int lanes_per = 32 / NV;
#pragma unroll
    for (int off = lanes_per / 2; off > 0; off >>= 1) r += __shfl_xor_sync(0xffffffffu, r, off);
    return r;
  }

  __device__ void attn_stage(int l) {
    constexpr int DPL = HD / 32;       // dims per lane
    constexpr int PPW = kKvTilePos / kConsumerWarps;  // positions per warp per tile (4)
    constexpr int NV = PPW * G;        // scores per warp per tile
    static_assert(NV <= 32 && (NV & (NV - 1)) == 0, "scores per warp must be a power of two <= 32");
    constexpr int LPV = 32 / NV;       // lanes per value after the reduction
    const float qscale = 1.4426950408889634f / sqrtf((float)HD);  // log2(e)/sqrt(hd)
    const unsigned row_bytes = HD * 2;
    const int NU = p.B * p.hkv * p.nch;
    for (int u = blockIdx.x; u < NU; u += gridDim.x) {
      AttnUnit a = attn_unit(p, m, u);
      // q heads of the group, pre-scaled
      float q[G][DPL];
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const uint16_t* qp = p.qbuf + (size_t)a.b * p.hq * HD + (size_t)(a.g * G + h) * HD + lane * DPL;
#pragma unroll
        for (int j = 0; j < DPL; ++j) q[h][j] = bf16f(ldcg_u16(qp + j)) * qscale;
      }
      float mrun[G], lrun[G], acc[G][DPL];
#pragma unroll
      for (int h = 0; h < G; ++h) {
        mrun[h] = -INFINITY;
        lrun[h] = 0.f;
#pragma unroll
        for (int j = 0; j < DPL; ++j) acc[h][j] = 0.f;
      }
      const int newpos = a.T - 1;
      for (int t = a.tile0; t < a.tile1; ++t) {
        const uint8_t* slot = wait_item();
        if (!dead) {
          const int p0 = t * kKvTilePos;
          const int npos = min(kKvTilePos, a.T - p0);
          float s[NV];
          const uint16_t* krow[PPW];
          const uint16_t* vrow[PPW];
#pragma unroll
          for (int i = 0; i < PPW; ++i) {
            const int j = warp * PPW + i;
            const int pa = p0 + j;
            if (pa == newpos) {
              krow[i] = p.kc + kv_row(p, l, a.b, a.g, pa);
              vrow[i] = p.vc + kv_row(p, l, a.b, a.g, pa);
            } else {
              krow[i] = reinterpret_cast<const uint16_t*>(slot + j * row_bytes);
              vrow[i] = reinterpret_cast<const uint16_t*>(slot + kKvTilePos * row_bytes + j * row_bytes);
            }
            float kf[DPL];
            if (j < npos) {
              if (pa == newpos) {
#pragma unroll
                for (int d = 0; d < DPL; ++d) kf[d] = bf16f(ldcg_u16(krow[i] + lane * DPL + d));
              } else {
#pragma unroll
                for (int d = 0; d < DPL; ++d) kf[d] = bf16f(krow[i][lane * DPL + d]);
              }
            } else {
#pragma unroll
              for (int d = 0; d < DPL; ++d) kf[d] = 0.f;
            }
#pragma unroll
            for (int h = 0; h < G; ++h) {
              float acc_s = 0.f;
#pragma unroll
              for (int d = 0; d < DPL; ++d) acc_s = fmaf(q[h][d], kf[d], acc_s);
              s[i * G + h] = acc_s;
            }
          }
          float mine = warp_transpose_reduce<NV>(s);
          const int vidx = lane / LPV;
          const int my_i = vidx / G, my_h = vidx % G;
          if (warp * PPW + my_i >= npos) mine = -INFINITY;
          // per-head maximum over this warp's positions: value index bits above log2(G)
          float bm = mine;
#pragma unroll
          for (int off = LPV * G; off < 32; off <<= 1) bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, off));
          float mnew[G], corr[G];
#pragma unroll
          for (int h = 0; h < G; ++h) {
            float bmh = __shfl_sync(0xffffffffu, bm, h * LPV);
            mnew[h] = fmaxf(mrun[h], bmh);
            corr[h] = (mnew[h] == -INFINITY) ? 1.f : exp2f(mrun[h] - mnew[h]);
          }
          float mn_own = mnew[0];
#pragma unroll
          for (int h = 1; h < G; ++h)
            if (my_h == h) mn_own = mnew[h];
          const float pown = (mine == -INFINITY) ? 0.f : exp2f(mine - mn_own);
          float pv[NV];
#pragma unroll
          for (int v = 0; v < NV; ++v) pv[v] = __shfl_sync(0xffffffffu, pown, v * LPV);
#pragma unroll
          for (int h = 0; h < G; ++h) {
            float ls = 0.f;
#pragma unroll
            for (int i = 0; i < PPW; ++i) ls += pv[i * G + h];
            lrun[h] = lrun[h] * corr[h] + ls;
            mrun[h] = mnew[h];
#pragma unroll
            for (int d = 0; d < DPL; ++d) acc[h][d] *= corr[h];
          }
#pragma unroll
          for (int i = 0; i < PPW; ++i) {
            const int j = warp * PPW + i;
            if (j < npos) {
              float vf[DPL];
              if (p0 + j == newpos) {
#pragma unroll
                for (int d = 0; d < DPL; ++d) vf[d] = bf16f(ldcg_u16(vrow[i] + lane * DPL + d));
              } else {
#pragma unroll
                for (int d = 0; d < DPL; ++d) vf[d] = bf16f(vrow[i][lane * DPL + d]);
              }
#pragma unroll
              for (int h = 0; h < G; ++h)
#pragma unroll
                for (int d = 0; d < DPL; ++d) acc[h][d] = fmaf(pv[i * G + h], vf[d], acc[h][d]);
            }
          }
        }
        release_item();
      }
      // merge the 8 warps' states: red = [warp][h][HD + 2]
      float* wst = red;
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float* r = wst + ((size_t)warp * G + h) * (HD + 2);
#pragma unroll
        for (int d = 0; d < DPL; ++d) r[lane * DPL + d] = acc[h][d];
        if (lane == 0) {
          r[HD] = mrun[h];
          r[HD + 1] = lrun[h];
        }
      }
      cons_sync();
      float* dst = p.attn_part + ((((size_t)a.b * p.hkv + a.g) * p.nch + a.c) * G) * (HD + 2);
      for (int idx = tid; idx < G * HD; idx += 256) {
        const int h = idx / HD, d = idx % HD;
        float M = -INFINITY;
        for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, wst[((size_t)w * G + h) * (HD + 2) + HD]);
        float A = 0.f, Lsum = 0.f;
        if (M != -INFINITY) {
          for (int w = 0; w < kConsumerWarps; ++w) {
            const float* r = wst + ((size_t)w * G + h) * (HD + 2);
            const float e = exp2f(r[HD] - M);
            A = fmaf(e, r[d], A);
            Lsum = fmaf(e, r[HD + 1], Lsum);
          }
        }
        dst[(size_t)h * (HD + 2) + d] = A;
        if (d == 0) {
          dst[(size_t)h * (HD + 2) + HD] = M;
          dst[(size_t)h * (HD + 2) + HD + 1] = Lsum;
        }
      }
      __threadfence();
      cons_sync();
      int* cnt = p.attn_cnt + (size_t)a.b * p.hkv + a.g;
      if (tid == 0) m->fin_old[0] = dead ? -1 : atom_add_acqrel(cnt, 1);
      cons_sync();
      if (m->fin_old[0] == p.nch - 1) {
        __threadfence();
        const float* src = p.attn_part + (((size_t)a.b * p.hkv + a.g) * p.nch * G) * (HD + 2);
        for (int idx = tid; idx < G * HD; idx += 256) {
          const int h = idx / HD, d = idx % HD;
          float M = -INFINITY;
          for (int c = 0; c < p.nch; ++c) M = fmaxf(M, ldcg(src + ((size_t)c * G + h) * (HD + 2) + HD));
          float A = 0.f, Lsum = 0.f;
          for (int c = 0; c < p.nch; ++c) {
            const float* r = src + ((size_t)c * G + h) * (HD + 2);
            const float mc = ldcg(r + HD);
            if (mc == -INFINITY) continue;
            const float e = exp2f(mc - M);
            A = fmaf(e, ldcg(r + d), A);
            Lsum = fmaf(e, ldcg(r + HD + 1), Lsum);
          }
          const float o = Lsum > 0.f ? A / Lsum : 0.f;
          p.obuf[(size_t)a.b * p.hq * HD + (size_t)(a.g * G + h) * HD + d] = f2bf(o);
        }
        if (tid == 0) atomicExch(cnt, 0);
      }
      cons_sync();
    }
  }

  // -------- the step --------

  __device__ void run() {
    trace();
    for (int l = 0; l < p.L; ++l) {
      const LayerDev& Ld = p.layers[l];
      // attention block
      stage_rmsnorm(l, nullptr, Ld.attn_norm);
      gemv_stage(K_QKV, l, 0);
      gsync(1);
      if (l == 0 && blockIdx.x == 0 && tid == 0 && !dead)
        for (int b = 0; b < p.B; ++b) p.lengths[p.seq0 + b] = m->len[b] + 1;
      attn_stage(l);
      gsync(2);
      stage_copy(p.obuf, p.hq * HD, (size_t)p.hq * HD, 0);
      cons_sync();
      gemv_stage(K_O, l, 0);
      gsync(3);
      // FFN block
      stage_rmsnorm(0, p.xmid, Ld.ffn_norm);
      int U = 0;
      if (p.dense) {
        gemv_stage(K_SHGU, l, 0);
      } else {
        gemv_stage(K_ROUTER, l, 0);
        if (p.nsh) gemv_stage(K_SHGU, l, 0);
        // routing result (published by the router's finaliser)
        if (tid == 0) {
          int Uv = 0;
          if (!dead && wait_flag(p, p.rt_flag + l, p.epoch, 12)) Uv = min(max(__ldcg(p.rt_u), 0), p.umax);
          else dead = true;
          m->U = Uv;
          m->flag = dead ? 0 : 1;
        }
        cons_sync();
        if (!m->flag) dead = true;
        U = m->U;
        for (int i = tid; i < U; i += 256) m->elist[i] = min(max(__ldcg(p.rt_elist + i), 0), p.E - 1);
        for (int i = tid; i < BM * kMaxExperts; i += 256) {
          int b = i / kMaxExperts, u = i % kMaxExperts;
          m->gate[b][u] = (b < p.B && u < U) ? __ldcg(p.rt_gate + (size_t)b * kMaxExperts + u) : 0.f;
        }
        cons_sync();
        gemv_stage(K_RTGU, l, U);
      }
      gsync(4);
      // down projections of all active experts, gate-weighted, + residual
      {
        const StageGeo g = stage_geo(p, K_D, U);
        const int t0 = range_lo(g.T, blockIdx.x, gridDim.x), t1 = range_lo(g.T, blockIdx.x + 1, gridDim.x);
        int v_lo = 0, v_hi = -1;
        if (t1 > t0) {
          v_lo = t0 / g.tpe;
          v_hi = (t1 - 1) / g.tpe;
        }
        if (tid == 0) m->v_lo = v_lo;
        for (int i = tid; i < BM; i += 256) m->gate[i][U] = 1.f;  // shared / dense expert
        for (int v = v_lo; v <= v_hi; ++v) {
          const uint16_t* src = (v < U) ? p.hrt + (size_t)v * p.MB * p.inter : p.hsh;
          stage_copy(src, p.inter, (size_t)p.inter, (v - v_lo) * p.inter);
        }
        cons_sync();
        gemv_stage(K_D, l, U);
      }
      gsync(5);
    }
    if (p.V > 0) {
      stage_rmsnorm(p.L, nullptr, p.final_norm);
      gemv_stage(K_LM, 0, 0);
    }
    trace();
  }
};

// ---------------------------------------------------------------------------------------------

template <int BM, int HD, int G>
__global__ void __launch_bounds__(kThreads, 1) decode_step_kernel(const __grid_constant__ KParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const SmemLayout L = smem_layout(p.ring, BM, p.xmax, HD, G);
  uint8_t* ring = smem + L.ring_off;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.full_off);
  uint64_t* empty = reinterpret_cast<uint64_t*>(smem + L.empty_off);
  uint16_t* xs = reinterpret_cast<uint16_t*>(smem + L.xs_off);
  float* red = reinterpret_cast<float*>(smem + L.red_off);
  Misc* m = reinterpret_cast<Misc*>(smem + L.misc_off);

  const int tid = threadIdx.x;
  if (tid == 0) {
    for (int s = 0; s < p.ring; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (tid < kMaxBatch) {
    int len = 0, tok = 0;
    if (tid < p.B) {
      len = p.lengths[p.seq0 + tid];
      if (len < 0 || len >= p.max_ctx) {
        raise_err(p, kDevBadArg, 1);
        len = 0;
      }
      if (p.tokens) {
        tok = p.tokens[tid];
        if (tok < 0 || tok >= p.V) {
          raise_err(p, kDevBadArg, 2);
          tok = 0;
        }
      }
    }
    m->len[tid] = len;
    m->tok[tid] = tok;
  }
  __syncthreads();

  if (tid >= kConsumerWarps * 32) {
    if (tid == kConsumerWarps * 32) {
      Producer<BM, HD, G> prod(p, ring, full, empty, m);
      prod.run();
    }
    return;
  }
  Consumer<BM, HD, G> cons(p, ring, full, empty, xs, red, m);
  cons.run();
}

}  // namespace dec
