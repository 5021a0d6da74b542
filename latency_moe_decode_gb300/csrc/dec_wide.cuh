// The decode step for 9 .. 64 tokens (sequences side by side): the tensor-core expert GEMMs of a
// batched decode ("vLLM's Kimi K3 Backend Hits 842 Tokens per Second", section "A narrow
// deployment lane": decode batches up to 64; section "Throughput holds across the tested range").
//
// At these batches every layer streams most of its routed experts (a 64-token step selects ~all
// 64), so a step is long and a cross-CTA hop is cheap beside it. The kernel therefore runs each
// layer as a fixed sequence of phases separated by grid barriers (one releasing arrival per CTA
// on a counter, bounded polls), and keeps every GEMV stage's input in global memory as the
// tensor cores' B operand: per k block of 128 activations, nr rows of E4M3 pieces (token t's two
// pieces in rows 2t, 2t + 1) plus one exponent byte per token. The producer warp copies a weight
// tile and the B block of its k block into one ring slot; the MMA warp multiplies them with
// tcgen05.mma kind::f8f6f4 (M = 128 weight rows, N = nr, K = 128) into a TMEM slice; the consumer
// warps scale each tile's product (block scale, the pieces' exponent) into fp32 registers and
// write one split-K partial per output row block. Routed experts multiply every token of the step
// (the MMA costs the same for any N <= 128) and keep only their routed tokens' rows.
//
// Phases of a layer (barrier after each):
//   q/k/v GEMV | attention (each unit sums its q/k/v partials, applies RoPE, appends its key and
//   value, streams its KV tiles) | chunk merge -> B blocks of the attention output | output
//   projection GEMV | x_mid = x + projection, RMSNorm -> B blocks | router and shared expert
//   gate/up GEMVs | routing (one CTA per token) | routed gate/up GEMV | SwiGLU -> B blocks per
//   expert slot | down GEMV (expert-major, gate applied per partial) | layer output, next RMSNorm
//   -> B blocks.
// Then the LM head GEMV, its finalisation (logits, argmax) and the next tokens.
#pragma once
#include "dec_kernel.cuh"

namespace dec {
namespace wide {

constexpr int kGC = 256;           // TMEM columns per group of tile products
constexpr int kNGW = 2;            // groups in flight (all 512 columns)
constexpr int kBarsPerLayer = 11;  // grid barriers of one layer

// ring slot: slot_tiles weight tiles, then their B blocks (a 32 KB hand-off per slot at most)
__host__ __device__ constexpr int slot_tiles(int nr) { return nr >= 128 ? 1 : 2; }
__host__ __device__ constexpr int slot_bytes(int nr) { return slot_tiles(nr) * (kTileBytes + nr * 128); }

// Partial-sum slots reserved per segment (output row block) of kbs tiles when a stage of T tiles
// is split into contiguous ranges over G CTAs: with T < G every tile has its own CTA; otherwise a
// range holds at least T / G tiles, so a segment meets at most ceil(kbs / (T / G)) + 1 ranges.
__host__ __device__ inline int seg_slots(int T, int kbs, int G) {
  if (T < G) return kbs;
  const int per = T / G;
  const int b = (kbs + per - 1) / per + 1;
  return b < kbs ? b : kbs;
}

struct WGeo {
  int T;    // tiles
  int kbs;  // tiles per segment (one output row block's k blocks)
  int tpe;  // expert stages: tiles of one expert slot
  int S;    // partial slots per segment
};
// Routed gate/up: U expert slots x n_rb_gu row blocks x kb_d k blocks. Down: U + n_shared slots
// (the shared expert last), expert major, segment (u, rb) = its kb_i k blocks.
__host__ __device__ inline WGeo wgeo(const KParams& p, int kind, int U, int G) {
  WGeo g;
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
  g.S = seg_slots(g.T, g.kbs, G);
  return g;
}

// attention work units: (token b, KV head g, context chunk c)
struct WUnit {
  int b, g, c, tile0, tile1, T;
};

struct WMisc {
  const unsigned* wt_addr[1];  // grid barrier poll (warp 0)
  unsigned wt_want[1];
  uint64_t rt_bar;    // consumers -> producer and MMA warp: the layer's routing is in elist / U
  uint64_t mma_done;  // the MMA warp's last MMAs are done (TMEM may be freed)
  uint64_t tm_ready;  // TMEM allocated
  // consumers -> MMA warp: GEMV stages begun so far (a count, so that the consumers may start
  // several stages in a row without the MMA warp losing track). The MMA warp skips the
  // attention's KV items without waiting for them; a slot's next phase may only be waited for
  // once its previous one has completed (a parity wait one phase early reports completion), and
  // the consumers start a stage only after consuming every KV item before it.
  unsigned stages_begun;
  uint64_t tfull[kNGW], tempty[kNGW];
  float2 hdr[kNGW][8];  // block scales of each group's tiles (the slots may be refilled first)
  uint32_t tmem_base;
  int flag;
  int U;       // distinct routed experts of the layer
  int npairs;  // (expert slot, token) pairs of the SwiGLU phase
  int elist[kMaxExperts];
  int len[kWideMax];
  int tok[kWideMax];
  unsigned long long umask[kMaxExperts + 1];  // tokens routed to expert slot u (slot U: shared)
  uint8_t wsel[kWideMax][16];                 // expert slot of each token's selections
  float wgate[kWideMax][16];                  // and their gates
  float rsum[kConsumerWarps];
  alignas(16) int8_t ex[kMaxKb * kWideMax];  // exponents of the running GEMV stage's B blocks [row][token]
};

struct WLayout {
  int ring_off, full_off, empty_off, mempty_off, red_off, misc_off, total;
};
__host__ __device__ inline WLayout wlayout(int ring, int nr, int hd, int group) {
  WLayout s;
  s.ring_off = 0;
  s.full_off = align_up(ring * slot_bytes(nr), 128);
  s.empty_off = s.full_off + ring * 8;
  s.mempty_off = s.empty_off + ring * 8;
  s.red_off = align_up(s.mempty_off + ring * 8, 128);
  int red = kConsumerWarps * group * (hd + 2) * 4;       // attention: the warps' states
  red = red > 2 * (group + 2) * hd * 4 ? red : 2 * (group + 2) * hd * 4;  // the unit's q/k/v
  const int pairs = (kMaxExperts + kWideMax * 17) * 4;   // routing marks, SwiGLU pairs
  red = red > pairs ? red : pairs;
  s.misc_off = align_up(s.red_off + red, 128);
  s.total = align_up(s.misc_off + (int)sizeof(WMisc), 128);
  return s;
}

__device__ __forceinline__ WUnit wunit(const KParams& p, const WideParams& w, const WMisc* m, int u) {
  WUnit a;
  const int per_b = p.hkv * w.nch;
  a.b = u / per_b;
  a.g = (u / w.nch) % p.hkv;
  a.c = u % w.nch;
  a.T = m->len[a.b] + 1;
  const int ntile = (a.T + kKvTilePos - 1) / kKvTilePos;
  const int tpc = (ntile + w.nch - 1) / w.nch;
  a.tile0 = min(ntile, a.c * tpc);
  a.tile1 = min(ntile, a.tile0 + tpc);
  return a;
}

// byte of (row, column c) in a B block: 8-row groups 1024 bytes apart, 16-byte chunks of a row
// 128 bytes apart, rows of a core matrix 16 bytes apart
__device__ __forceinline__ int boff(int row, int c) { return (row >> 3) * 1024 + (c >> 4) * 128 + (row & 7) * 16 + (c & 15); }

__device__ __forceinline__ float* part_of(const KParams& p, int kind) {
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

// ---------------------------------------------------------------------------------------------
// producer warp (one thread): weight tiles and their B blocks, KV tiles

template <int NR, int HD, int G>
struct WProducer {
  static constexpr int ST = slot_tiles(NR), PBS = NR * 128, SB = slot_bytes(NR);
  const KParams& p;
  const WideParams& w;
  uint8_t* ring;
  uint64_t* full;
  uint64_t* empty;
  uint64_t* mempty;
  WMisc* m;
  unsigned item = 0;
  int pslot = 0;
  unsigned plap = 0;
  unsigned landed = 0;
  int lslot = 0;
  unsigned llap = 0;
  // per slot (one bit each): whether its last use completes mempty (the MMA warp's commit) or
  // empty (the consumer warps), and the parity of each kind's uses so far
  uint32_t last_mma = 0, ne_par = 0, nm_par = 0;
  uint64_t pol_stream = 0, pol_near = 0;
  bool dead = false;
  unsigned lay = 0;

  __device__ WProducer(const KParams& p_, const WideParams& w_, uint8_t* r, uint64_t* f, uint64_t* e, uint64_t* me,
                       WMisc* m_)
      : p(p_), w(w_), ring(r), full(f), empty(e), mempty(me), m(m_) {}

  __device__ __forceinline__ static bool within(const void* src, size_t bytes, const void* base, size_t extent) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(src), b = reinterpret_cast<uintptr_t>(base);
    return a >= b && a + bytes <= b + extent && (a & 15u) == 0 && (bytes & 15u) == 0;
  }

  // the next slot, once at most p.inflight - 1 copies are in flight and its last use is over
  __device__ bool claim(int& slot, bool mma_use) {
    while (item - landed >= (unsigned)p.inflight) {
      if (!mbar_wait(&full[lslot], llap & 1, p, 42)) {
        dead = true;
        return false;
      }
      ++landed;
      if (++lslot == p.ring) {
        lslot = 0;
        ++llap;
      }
    }
    slot = pslot;
    const uint32_t bit = 1u << slot;
    if (plap > 0) {
      const bool pm = (last_mma & bit) != 0;
      const unsigned par = (((pm ? nm_par : ne_par) >> slot) & 1u) ^ 1u;
      if (!mbar_wait(pm ? &mempty[slot] : &empty[slot], par, p, 43)) {
        dead = true;
        return false;
      }
    }
    if (mma_use) {
      last_mma |= bit;
      nm_par ^= bit;
    } else {
      last_mma &= ~bit;
      ne_par ^= bit;
    }
    return true;
  }
  __device__ __forceinline__ void advance() {
    ++item;
    if (++pslot == p.ring) {
      pslot = 0;
      ++plap;
    }
  }

  // Wait (bounded) until every CTA has passed grid barrier k, then order the bulk copies that
  // follow (async proxy) after the data those CTAs wrote before it.
  __device__ bool wait_bar(unsigned k) {
    if (dead) return false;
    const unsigned want = k * gridDim.x;
    const unsigned long long t0 = gtimer();
    for (unsigned it = 1; ld_acquire(w.bar) < want; ++it) {
      if ((it & 15u) == 0) {
        if (aborted(p)) {
          dead = true;
          return false;
        }
        if (gtimer() - t0 > p.timeout_ns) {
          raise_err(p, kDevTimeout, 44);
          dead = true;
          return false;
        }
      }
    }
    fence_proxy_async_global();
    return true;
  }

  __device__ const uint8_t* tile_src(int kind, const LayerDev& Ld, const WGeo& g, int t, int U, const int* elist) const {
    switch (kind) {
      case K_QKV: return Ld.qkv + (size_t)t * kTileBytes;
      case K_O: return Ld.o + (size_t)t * kTileBytes;
      case K_ROUTER: return Ld.router + (size_t)t * kTileBytes;
      case K_SHGU: return Ld.sh_gu + (size_t)t * kTileBytes;
      case K_RTGU: {
        const int u = t / g.tpe;
        return Ld.e_gu + (size_t)elist[u] * p.e_gu_stride + (size_t)(t - u * g.tpe) * kTileBytes;
      }
      case K_D: {
        const int u = t / g.tpe;
        const uint8_t* base = u < U ? Ld.e_d + (size_t)elist[u] * p.e_d_stride : Ld.sh_d;
        return base + (size_t)(t - u * g.tpe) * kTileBytes;
      }
      default: return p.lm + (size_t)t * kTileBytes;
    }
  }
  __device__ const uint8_t* b_src(int kind, const WGeo& g, int t) const {
    const int kb = t % g.kbs;
    if (kind == K_O) return w.pbo + (size_t)kb * PBS;
    if (kind == K_D) return w.pbh + ((size_t)(t / g.tpe) * p.kb_i + kb) * PBS;
    return w.pbx + (size_t)kb * PBS;
  }

  __device__ void issue_gemv(int kind, int l, int U, const int* elist) {
    if (dead) return;
    const WGeo g = wgeo(p, kind, U, gridDim.x);
    const int t0 = range_lo(g.T, blockIdx.x, gridDim.x), t1 = range_lo(g.T, blockIdx.x + 1, gridDim.x);
    const LayerDev& Ld = p.layers[l < p.L ? l : 0];
    for (int t = t0; t < t1; t += ST) {
      int slot;
      if (!claim(slot, true)) return;
      const int n = min(ST, t1 - t);
      const uint8_t* a[ST];
      const uint8_t* b[ST];
      bool ok = true;
#pragma unroll
      for (int j = 0; j < ST; ++j) {
        if (j < n) {
          a[j] = tile_src(kind, Ld, g, t + j, U, elist);
          b[j] = b_src(kind, g, t + j);
          ok = ok && within(a[j], kTileBytes, p.warena, p.warena_bytes) && within(b[j], PBS, w.pb, w.pb_bytes);
        }
      }
      uint8_t* dst = ring + (size_t)slot * SB;
      if (!ok) {
        raise_err(p, kDevBadArg, 45);
        mbar_arrive(&full[slot]);
        advance();
        continue;
      }
      mbar_arrive_expect_tx(&full[slot], (unsigned)n * (kTileBytes + PBS));
      if (n == 2 && a[ST - 1] == a[0] + kTileBytes) {
        bulk_g2s_hint(dst, a[0], 2 * kTileBytes, &full[slot], pol_stream);
      } else {
        for (int j = 0; j < n; ++j) bulk_g2s_hint(dst + (size_t)j * kTileBytes, a[j], kTileBytes, &full[slot], pol_stream);
      }
      uint8_t* bdst = dst + (size_t)ST * kTileBytes;
      if (n == 2 && b[ST - 1] == b[0] + PBS) {
        bulk_g2s_hint(bdst, b[0], 2 * PBS, &full[slot], pol_near);
      } else {
        for (int j = 0; j < n; ++j) bulk_g2s_hint(bdst + (size_t)j * PBS, b[j], PBS, &full[slot], pol_near);
      }
      advance();
    }
  }

  // KV tiles of the CTA's attention units (rows before the new position: written by earlier
  // launches; the unit patches the new position into its copy)
  __device__ void issue_attn(int l) {
    if (dead) return;
    const int NU = p.B * p.hkv * w.nch;
    const unsigned row_bytes = HD * 2;
    for (int u = blockIdx.x; u < NU; u += gridDim.x) {
      const WUnit a = wunit(p, w, m, u);
      for (int t = a.tile0; t < a.tile1; ++t) {
        int slot;
        if (!claim(slot, false)) return;
        const int p0 = t * kKvTilePos;
        const int n = min(kKvTilePos, a.T - p0);
        uint8_t* dst = ring + (size_t)slot * SB;
        const size_t r0 = kv_row(p, l, a.b, a.g, p0);
        if (n < 1 || n > kKvTilePos || !within(p.kc + r0, n * row_bytes, p.kc, p.kv_bytes) ||
            !within(p.vc + r0, n * row_bytes, p.vc, p.kv_bytes)) {
          raise_err(p, kDevBadArg, 46);
          mbar_arrive(&full[slot]);
          advance();
          continue;
        }
        mbar_arrive_expect_tx(&full[slot], 2u * n * row_bytes);
        bulk_g2s_hint(dst, p.kc + r0, n * row_bytes, &full[slot], pol_near);
        bulk_g2s_hint(dst + kKvTilePos * row_bytes, p.vc + r0, n * row_bytes, &full[slot], pol_near);
        advance();
      }
    }
  }

  __device__ bool routing(int& U, int* elist) {
    if (dead) return false;
    if (!mbar_wait(&m->rt_bar, lay & 1u, p, 47)) {
      dead = true;
      return false;
    }
    U = min(max(m->U, 0), w.hmax - p.nsh);
    for (int i = 0; i < U; ++i) elist[i] = min(max(m->elist[i], 0), p.E - 1);
    return true;
  }

  __device__ void drain() {
    const unsigned first = item > (unsigned)p.ring ? item - p.ring : 0u;
    for (unsigned i = first; i < item; ++i) {
      const int slot = i % p.ring;
      const unsigned par = (i / p.ring) & 1;
      const unsigned long long t0 = gtimer();
      while (!mbar_try_wait(&full[slot], par)) {
        if (gtimer() - t0 > p.timeout_ns) break;
      }
    }
  }

  // The load program. A GEMV stage's copies start once the barrier after the phase that wrote
  // its B blocks has passed; KV tiles need no barrier.
  __device__ void run() {
    int elist[kMaxExperts];
    pol_stream = l2_policy(true);
    pol_near = l2_policy(false);
#pragma unroll 1
    for (int l = 0; l < p.L && !dead; ++l) {
      const unsigned base = 1u + (unsigned)(kBarsPerLayer * l);
      if (!wait_bar(base)) break;
      issue_gemv(K_QKV, l, 0, elist);
      issue_attn(l);
      if (!wait_bar(base + 3)) break;
      issue_gemv(K_O, l, 0, elist);
      if (!wait_bar(base + 5)) break;
      if (!p.dense) issue_gemv(K_ROUTER, l, 0, elist);
      if (p.dense || p.nsh) issue_gemv(K_SHGU, l, 0, elist);
      int U = 0;
      if (!p.dense) {
        if (!routing(U, elist)) break;
        issue_gemv(K_RTGU, l, U, elist);
      }
      if (!wait_bar(base + 9)) break;
      issue_gemv(K_D, l, U, elist);
      ++lay;
    }
    if (p.V > 0 && !dead && wait_bar(1u + (unsigned)(kBarsPerLayer * p.L))) issue_gemv(K_LM, 0, 0, elist);
    drain();
  }
};

// ---------------------------------------------------------------------------------------------
// MMA warp (one thread): the CTA's tiles in the consumers' order, in groups of up to GT tiles of
// one segment per TMEM group (kGC columns), kNGW groups in flight.

template <int NR, int HD, int G>
struct WMma {
  static constexpr int ST = slot_tiles(NR), PBS = NR * 128, SB = slot_bytes(NR), GT = kGC / NR;
  const KParams& p;
  const WideParams& w;
  uint8_t* ring;
  uint64_t* full;
  uint64_t* mempty;
  WMisc* m;
  int slot = 0;
  unsigned lap = 0;
  unsigned gseq = 0;
  unsigned stage = 0;  // GEMV stages reached
  bool dead = false;
  uint32_t tmem = 0;
  unsigned lay = 0;

  __device__ WMma(const KParams& p_, const WideParams& w_, uint8_t* r, uint64_t* f, uint64_t* me, WMisc* m_)
      : p(p_), w(w_), ring(r), full(f), mempty(me), m(m_) {}

  __device__ __forceinline__ void skip(int n) {
    for (int i = 0; i < n; ++i)
      if (++slot == p.ring) {
        slot = 0;
        ++lap;
      }
  }

  // wait (bounded) until the consumers have begun GEMV stage number `stage` (1-based)
  __device__ void wait_stage() {
    if (dead) return;
    const unsigned long long t0 = gtimer();
    for (unsigned it = 1; *reinterpret_cast<volatile unsigned*>(&m->stages_begun) < stage; ++it) {
      if ((it & 63u) == 0) {
        if (aborted(p)) {
          dead = true;
          return;
        }
        if (gtimer() - t0 > p.timeout_ns) {
          raise_err(p, kDevTimeout, 56);
          dead = true;
          return;
        }
      }
    }
    __threadfence_block();
  }

  __device__ void gemv(int kind, int U) {
    ++stage;
    wait_stage();
    const WGeo g = wgeo(p, kind, U, gridDim.x);
    const int t0 = range_lo(g.T, blockIdx.x, gridDim.x), t1 = range_lo(g.T, blockIdx.x + 1, gridDim.x);
    constexpr uint32_t idesc = idesc_e4m3_f32(kTileRows, NR);
    int j = 0;
#pragma unroll 1
    for (int t = t0; t < t1;) {
      const int seg = t / g.kbs;
      const int n = min(GT, min(t1, (seg + 1) * g.kbs) - t);
      const int gsl = gseq % kNGW;
      if (!dead && gseq >= (unsigned)kNGW && !mbar_wait(&m->tempty[gsl], (gseq / kNGW - 1) & 1, p, 48)) dead = true;
#pragma unroll 1
      for (int i = 0; i < n; ++i, ++t) {
        if (!dead && j == 0 && !mbar_wait(&full[slot], lap & 1, p, 49)) dead = true;
        const uint8_t* a = ring + (size_t)slot * SB + (size_t)j * kTileBytes;
        const uint8_t* b = ring + (size_t)slot * SB + (size_t)ST * kTileBytes + (size_t)j * PBS;
        if (!dead) {
          tc_fence_after();
          m->hdr[gsl][i] = *reinterpret_cast<const float2*>(a + kTileData);
          const uint64_t ad = smem_desc(a, 128, 1024), bd = smem_desc(b, 128, 1024);
          const uint32_t d = tmem + (uint32_t)(gsl * kGC + i * NR);
#pragma unroll
          for (int k = 0; k < kTileK / 32; ++k)
            mma_e4m3(d, ad + (uint64_t)(k * 16), bd + (uint64_t)(k * 16), idesc, k > 0 ? 1u : 0u);
        }
        if (++j == ST || t == t1 - 1) {
          if (!dead) mma_commit(&mempty[slot]);
          j = 0;
          skip(1);
        }
      }
      if (!dead) {
        mma_commit(&m->tfull[gsl]);
        mbar_arrive(&m->tfull[gsl]);
      }
      ++gseq;
    }
  }

  __device__ void run() {
    if (!mbar_wait(&m->tm_ready, 0, p, 50)) dead = true;
    tc_fence_after();
    tmem = m->tmem_base;
#pragma unroll 1
    for (int l = 0; l < p.L; ++l) {
      gemv(K_QKV, 0);
      int items = 0;
      for (int u = blockIdx.x; u < p.B * p.hkv * w.nch; u += gridDim.x) {
        const WUnit a = wunit(p, w, m, u);
        items += a.tile1 - a.tile0;
      }
      skip(items);
      gemv(K_O, 0);
      if (!p.dense) gemv(K_ROUTER, 0);
      if (p.dense || p.nsh) gemv(K_SHGU, 0);
      int U = 0;
      if (!p.dense) {
        if (!dead && !mbar_wait(&m->rt_bar, lay & 1u, p, 51)) dead = true;
        U = min(max(m->U, 0), w.hmax - p.nsh);
        gemv(K_RTGU, U);
      }
      gemv(K_D, U);
      ++lay;
    }
    if (p.V > 0) gemv(K_LM, 0);
    if (gseq > 0) {
      const unsigned last = gseq - 1;
      const unsigned long long t0 = gtimer();
      while (!mbar_try_wait(&m->tfull[last % kNGW], (last / kNGW) & 1) && gtimer() - t0 < p.timeout_ns) {
      }
    }
    mbar_arrive(&m->mma_done);
  }
};

// ---------------------------------------------------------------------------------------------
// consumer warps

template <int NR, int HD, int G>
struct WConsumer {
  static constexpr int ST = slot_tiles(NR), PBS = NR * 128, SB = slot_bytes(NR), GT = kGC / NR;
  static constexpr int TPT = NR / 4;  // tokens per thread in a tile's epilogue
  static constexpr int MAXV = kMaxHidden / (kConsumerWarps * 32 * 8);  // 8-element chunks per thread
  const KParams& p;
  const WideParams& w;
  uint8_t* ring;
  uint64_t* full;
  uint64_t* empty;
  float* red;
  WMisc* m;
  unsigned item = 0;
  int rslot = 0;
  unsigned rpar = 0;
  bool dead = false;
  int warp, lane, tid;
  unsigned gseq = 0;  // tile groups handed over so far
  unsigned nbar = 0;  // grid barriers passed
  unsigned nstage = 0;  // GEMV stages begun (thread 0)
  uint32_t tmem = 0;

  __device__ WConsumer(const KParams& p_, const WideParams& w_, uint8_t* r, uint64_t* f, uint64_t* e, float* rd,
                       WMisc* m_)
      : p(p_), w(w_), ring(r), full(f), empty(e), red(rd), m(m_) {
    tid = threadIdx.x;
    warp = tid >> 5;
    lane = tid & 31;
  }

  __device__ const uint8_t* wait_item() {
    if (!dead && !mbar_wait(&full[rslot], rpar, p, 52)) dead = true;
    return ring + (size_t)rslot * SB;
  }
  __device__ void release_item() {
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[rslot]);
    ++item;
    if (++rslot == p.ring) {
      rslot = 0;
      rpar ^= 1;
    }
  }
  __device__ void ring_skip(int n) {
    for (int i = 0; i < n; ++i) {
      ++item;
      if (++rslot == p.ring) {
        rslot = 0;
        rpar ^= 1;
      }
    }
  }

  // Grid barrier: the CTA barrier orders every consumer thread's writes before the publishing
  // thread's releasing arrival; warp 0 polls (acquire, bounded) until all CTAs have arrived.
  __device__ void gbar() {
    ++nbar;
    cons_sync();
    if (tid == kPubThread && !dead) red_release_add(reinterpret_cast<int*>(w.bar), 1);
    if (warp == 0) {
      int ok = dead ? 0 : 1;
      if (ok) {
        if (lane == 0) {
          m->wt_addr[0] = w.bar;
          m->wt_want[0] = nbar * gridDim.x;
        }
        __syncwarp();
        ok = poll_all_geq(m->wt_addr, m->wt_want, 1, p.err, p.timeout_ns, 53);
      }
      if (lane == 0) m->flag = ok;
    }
    dead = cons_any(dead) || !m->flag;
  }

  // ---- B blocks

  // Pieces of activations c .. c + 7 of one k block (the half-warp's 16 chunks hold its 128) of
  // token t: with 2^a putting the block's largest |x| in [128, 256), x * 2^a = p1 + p2 / 16,
  // p1 = E4M3(x * 2^a), p2 = E4M3(16 (x * 2^a - p1)), rows 2t and 2t + 1 of block blk; the
  // exponent a goes to *ex. Called by whole warps.
  __device__ void pack8(uint8_t* blk, int8_t* ex, int t, int c, const float (&f)[8], bool in) {
    float mx = 0.f;
    if (in)
#pragma unroll
      for (int i = 0; i < 8; ++i) mx = fmaxf(mx, fabsf(f[i]));
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (!in) return;
    const int e = mx > 0.f ? (int)((__float_as_uint(mx) >> 23) & 0xFF) - 127 : 7;
    const int a = max(-120, min(120, 7 - e));
    const float sa = __int_as_float((127 + a) << 23);
    uint32_t w1[2], w2[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const float x0 = f[4 * i] * sa, x1 = f[4 * i + 1] * sa, x2 = f[4 * i + 2] * sa, x3 = f[4 * i + 3] * sa;
      const uint16_t q01 = float2_to_e4m3x2(x0, x1), q23 = float2_to_e4m3x2(x2, x3);
      const float2 g01 = e4m3x2_to_float2(q01), g23 = e4m3x2_to_float2(q23);
      const uint16_t r01 = float2_to_e4m3x2((x0 - g01.x) * 16.f, (x1 - g01.y) * 16.f);
      const uint16_t r23 = float2_to_e4m3x2((x2 - g23.x) * 16.f, (x3 - g23.y) * 16.f);
      w1[i] = (uint32_t)q01 | ((uint32_t)q23 << 16);
      w2[i] = (uint32_t)r01 | ((uint32_t)r23 << 16);
    }
    *reinterpret_cast<uint2*>(blk + boff(2 * t, c)) = make_uint2(w1[0], w1[1]);
    *reinterpret_cast<uint2*>(blk + boff(2 * t + 1, c)) = make_uint2(w2[0], w2[1]);
    if ((lane & 15) == 0) *ex = (int8_t)a;
  }
  // The same for a whole warp holding one k block, four activations c .. c + 3 per lane.
  __device__ void pack4(uint8_t* blk, int8_t* ex, int t, int c, const float (&f)[4]) {
    float mx = fmaxf(fmaxf(fabsf(f[0]), fabsf(f[1])), fmaxf(fabsf(f[2]), fabsf(f[3])));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    const int e = mx > 0.f ? (int)((__float_as_uint(mx) >> 23) & 0xFF) - 127 : 7;
    const int a = max(-120, min(120, 7 - e));
    const float sa = __int_as_float((127 + a) << 23);
    const float x0 = f[0] * sa, x1 = f[1] * sa, x2 = f[2] * sa, x3 = f[3] * sa;
    const uint16_t q01 = float2_to_e4m3x2(x0, x1), q23 = float2_to_e4m3x2(x2, x3);
    const float2 g01 = e4m3x2_to_float2(q01), g23 = e4m3x2_to_float2(q23);
    const uint16_t r01 = float2_to_e4m3x2((x0 - g01.x) * 16.f, (x1 - g01.y) * 16.f);
    const uint16_t r23 = float2_to_e4m3x2((x2 - g23.x) * 16.f, (x3 - g23.y) * 16.f);
    *reinterpret_cast<uint32_t*>(blk + boff(2 * t, c)) = (uint32_t)q01 | ((uint32_t)q23 << 16);
    *reinterpret_cast<uint32_t*>(blk + boff(2 * t + 1, c)) = (uint32_t)r01 | ((uint32_t)r23 << 16);
    if (lane == 0) *ex = (int8_t)a;
  }

  // Token t's row v (bf16, this thread's chunks k = (tid + j * 256) * 8) -> bf16(rmsnorm(v) * wn)
  // as B blocks of pbx. Called by the whole CTA.
  __device__ void norm_pack(int t, const uint4 (&v)[MAXV], const uint16_t* wn) {
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < MAXV; ++j) {
      const int k = (tid + j * kConsumerWarps * 32) * 8;
      if (k < p.d) {
        const uint32_t* u = reinterpret_cast<const uint32_t*>(&v[j]);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float a = bf16lo(u[q]), c = bf16hi(u[q]);
          ss = fmaf(a, a, ss);
          ss = fmaf(c, c, ss);
        }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (lane == 0) m->rsum[warp] = ss;
    cons_sync();
    float tot = 0.f;
#pragma unroll
    for (int wi = 0; wi < kConsumerWarps; ++wi) tot += m->rsum[wi];
    const float inv = 1.0f / sqrtf(tot / (float)p.d + p.eps);
#pragma unroll
    for (int j = 0; j < MAXV; ++j) {
      const int k = (tid + j * kConsumerWarps * 32) * 8;
      const bool in = k < p.d;  // (whole half-warps: d is a multiple of 128)
      float f[8];
      if (in) {
        const uint4 wv = __ldg(reinterpret_cast<const uint4*>(wn + k));
        const uint32_t* u = reinterpret_cast<const uint32_t*>(&v[j]);
        const uint32_t* wu = reinterpret_cast<const uint32_t*>(&wv);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          f[2 * q] = bf16f(f2bf((bf16lo(u[q]) * inv) * bf16lo(wu[q])));
          f[2 * q + 1] = bf16f(f2bf((bf16hi(u[q]) * inv) * bf16hi(wu[q])));
        }
      }
      const int kb = in ? k / kTileK : 0;
      pack8(w.pbx + (size_t)kb * PBS, w.exx + (size_t)kb * kWideMax + t, t, k % kTileK, f, in);
    }
    cons_sync();  // (m->rsum is reused by the next token)
  }

  // ---- GEMV stages

  // Add the products of group gs (n consecutive tiles of one segment, from tile t) into the
  // thread's accumulators: thread (warp w, lane) holds weight row 32 (w & 3) + lane of tokens
  // TPT (w >> 2) + j; token b's pieces are columns 2b, 2b + 1 of the tile's TMEM slice. Each
  // product is scaled by the tile's block scale and the pieces' 2^-a.
  __device__ __forceinline__ void epilogue(unsigned gs, int n, int kind, const WGeo& g, int t, int u_lo, float (&acc)[TPT]) {
    const int gsl = gs % kNGW;
    if (!dead && !mbar_wait(&m->tfull[gsl], (gs / kNGW) & 1, p, 54)) dead = true;
    dead = __any_sync(0xffffffffu, dead);  // (the TMEM loads below are warp-collective)
    const int q = warp & 3, h = warp >> 2, row = 32 * q + lane;
    if (!dead && h * TPT < p.B) {  // (warp-uniform)
      tc_fence_after();
#pragma unroll 1
      for (int i = 0; i < n; ++i, ++t) {
        const int kb = t % g.kbs;
        const int xr = kind == K_D ? (t / g.tpe - u_lo) * p.kb_i + kb : kb;
        const int8_t* ex = m->ex + xr * kWideMax + h * TPT;
        const float2 sc = m->hdr[gsl][i];
        const float s_r = row < 64 ? sc.x : sc.y;
        const uint32_t ta = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(gsl * kGC + i * NR + h * (NR / 2));
        // 16 columns (8 tokens) per load
#pragma unroll
        for (int c = 0; c < NR / 32; ++c) {
          float d[16];
          tmem_ld16(ta + 16 * c, d);
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float inv = __int_as_float((127 - (int)ex[8 * c + j]) << 23);
            acc[8 * c + j] = fmaf(s_r * inv, fmaf(d[2 * j + 1], 0.0625f, d[2 * j]), acc[8 * c + j]);
          }
        }
      }
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&m->tempty[gsl]);
  }

  __device__ float gate_of(int t, int u) const {
    for (int k = 0; k < p.topk; ++k)
      if (m->wsel[t][k] == u) return m->wgate[t][k];
    return 0.f;
  }

  // One segment's partial sums of the CTA: plain stores (read after the next grid barrier). The
  // routed stages keep only the tokens routed to the segment's expert slot; the down projection's
  // partials carry that token's gate.
  __device__ __forceinline__ void flush(int kind, const WGeo& g, int seg, int first, int U, const float (&acc)[TPT]) {
    if (dead) return;
    const int slot = contrib_slot(blockIdx.x, first, seg * g.kbs, g.T, gridDim.x);
    float* dst = part_of(p, kind) + (size_t)(seg * g.S + slot) * p.MB * kTileRows;
    const int row = 32 * (warp & 3) + lane, h = warp >> 2;
    int u = -1;
    unsigned long long mask = ~0ull;
    if (kind == K_RTGU) u = seg / p.n_rb_gu;
    if (kind == K_D) u = seg / p.n_rb_d;
    if (u >= 0) mask = m->umask[u];
    // (the thread's tokens h TPT + j: one base address, constant offsets)
    float* base = dst + (size_t)h * TPT * kTileRows + row;
    const unsigned long long mh = mask >> (h * TPT);
    const int nb = p.B - h * TPT;
#pragma unroll
    for (int j = 0; j < TPT; ++j) {
      if (j < nb && ((mh >> j) & 1ull)) {
        float v = acc[j];
        if (kind == K_D && u < U) v *= gate_of(h * TPT + j, u);
        base[j * kTileRows] = v;
      }
    }
  }

  __device__ void gemv(int kind, int U) {
    const WGeo g = wgeo(p, kind, U, gridDim.x);
    const int t0 = range_lo(g.T, blockIdx.x, gridDim.x), t1 = range_lo(g.T, blockIdx.x + 1, gridDim.x);
    // the exponents of the B blocks the CTA's tiles read (written before the last barrier)
    int u_lo = 0;
    if (t1 > t0 && !dead) {
      const int8_t* src;
      int rows;
      if (kind == K_D) {
        u_lo = t0 / g.tpe;
        const int u_hi = (t1 - 1) / g.tpe;
        rows = (u_hi - u_lo + 1) * p.kb_i;
        src = w.exh + (size_t)u_lo * p.kb_i * kWideMax;
      } else {
        rows = g.kbs;
        src = kind == K_O ? w.exo : w.exx;
      }
      if (rows > kMaxKb) {
        if (tid == 0) raise_err(p, kDevBadArg, 55);
        rows = 0;
      }
      for (int i = tid; i < rows * kWideMax / 16; i += kConsumerWarps * 32)
        reinterpret_cast<uint4*>(m->ex)[i] = ldcg4(src + (size_t)i * 16);
    }
    cons_sync();
    if (tid == 0) {  // (every earlier ring item has been consumed)
      ++nstage;
      __threadfence_block();
      *reinterpret_cast<volatile unsigned*>(&m->stages_begun) = nstage;
    }
    float acc[TPT];
    int seg_cur = -1, seg_first = 0;
#pragma unroll 1
    for (int t = t0;;) {
      const int seg = t < t1 ? t / g.kbs : -1;
      if (t == t1 || seg != seg_cur) {
        if (seg_cur >= 0) flush(kind, g, seg_cur, seg_first, U, acc);
        if (t == t1) break;
        seg_cur = seg;
        seg_first = t;
#pragma unroll
        for (int j = 0; j < TPT; ++j) acc[j] = 0.f;
      }
      const int n = min(GT, min(t1, (seg + 1) * g.kbs) - t);
      epilogue(gseq++, n, kind, g, t, u_lo, acc);
      t += n;
    }
    ring_skip((t1 - t0 + ST - 1) / ST);
    dead = cons_any(dead);
  }

  // ---- attention

  // The unit's q heads, key and value for its token: summed from the q/k/v partials, rotated
  // (half-split RoPE at the token's position), rounded to bf16; the unit whose chunk holds the
  // new position appends the key and value to the cache.
  __device__ void prologue(int l, const WUnit& a, float* qkvn) {
    const WGeo gq = wgeo(p, K_QKV, 0, gridDim.x);
    constexpr int NV_ = (G + 2) * HD;
    constexpr int NPT = (NV_ + kConsumerWarps * 32 - 1) / (kConsumerWarps * 32);
    float* raw = qkvn + NV_;
    const int pos = m->len[a.b];
    const size_t pst = (size_t)p.MB * kTileRows;
#pragma unroll
    for (int i = 0; i < NPT; ++i) {
      const int idx = tid + i * kConsumerWarps * 32;
      if (idx < NV_) {
        const int t = idx / HD, d = idx % HD;
        const int row = t < G ? (a.g * G + t) * HD + d : (t == G ? p.hq * HD : (p.hq + p.hkv) * HD) + a.g * HD + d;
        const int rb = row / kTileRows;
        const int nc = n_contrib(rb * gq.kbs, gq.kbs, gq.T, gridDim.x);
        const float* src = p.part_qkv + ((size_t)rb * gq.S * p.MB + a.b) * kTileRows + row % kTileRows;
        float s = 0.f;
#pragma unroll 1
        for (int c0 = 0; c0 < nc; c0 += 4) {
          float v[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) v[j] = c0 + j < nc ? ldcg(src + (size_t)(c0 + j) * pst) : 0.f;
#pragma unroll
          for (int j = 0; j < 4; ++j) s += v[j];
        }
        raw[idx] = s;
      }
    }
    cons_sync();
    const bool writer = (pos / kKvTilePos) >= a.tile0 && (pos / kKvTilePos) < a.tile1;
#pragma unroll
    for (int i = 0; i < NPT; ++i) {
      const int idx = tid + i * kConsumerWarps * 32;
      if (idx >= NV_) break;
      const int t = idx / HD, d = idx % HD;
      float val = raw[idx];
      if (t <= G) {
        const float2 cs = __ldg(p.rope + (size_t)pos * (HD / 2) + d % (HD / 2));
        const float other = raw[t * HD + (d < HD / 2 ? d + HD / 2 : d - HD / 2)];
        val = d < HD / 2 ? val * cs.x - other * cs.y : val * cs.x + other * cs.y;
      }
      const uint16_t bv = f2bf(val);
      qkvn[idx] = bf16f(bv);
      if (writer && t == G) p.kc[kv_row(p, l, a.b, a.g, pos) + d] = bv;
      if (writer && t == G + 1) p.vc[kv_row(p, l, a.b, a.g, pos) + d] = bv;
    }
    cons_sync();
  }

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
    constexpr int lanes_per = 32 / NV;
#pragma unroll
    for (int off = lanes_per / 2; off > 0; off >>= 1) r += __shfl_xor_sync(0xffffffffu, r, off);
    return r;
  }

  // Split-context GQA decode: unit (token b, KV head g, chunk c) over the KV tiles of its chunk
  // (each tile shared by the eight warps, 8 positions per warp, online softmax per warp, merged
  // per unit). One chunk: the normalised outputs go straight to the B blocks of the projection;
  // otherwise the chunk's state is published for the merge phase.
  __device__ void attention(int l) {
    constexpr int DPL = HD / 32;
    constexpr int PPW = kKvTilePos / kConsumerWarps;
    constexpr int NV = PPW * G;
    static_assert(NV <= 32 && (NV & (NV - 1)) == 0, "scores per warp must be a power of two <= 32");
    constexpr int LPV = 32 / NV;
    static_assert(DPL == 2 || DPL == 4, "head_dim 64 or 128");
    static_assert((G * HD) % kTileK == 0, "a KV group's heads must fill whole k blocks");
    const float qscale = 1.4426950408889634f / sqrtf((float)HD);
    const unsigned row_bytes = HD * 2;
    const int NU = p.B * p.hkv * w.nch;
#pragma unroll 1
    for (int u = blockIdx.x; u < NU; u += gridDim.x) {
      const WUnit a = wunit(p, w, m, u);
      float* qkvn = red;
      if (a.tile1 > a.tile0) prologue(l, a, qkvn);  // (CTA barriers inside: no branch on `dead`)
      float q[G][DPL];
#pragma unroll
      for (int h = 0; h < G; ++h)
#pragma unroll
        for (int j = 0; j < DPL; ++j) q[h][j] = qkvn[h * HD + lane * DPL + j] * qscale;
      float kn[DPL], vn[DPL];  // (the new key and value, patched into the tile that holds them)
      float mrun[G], lrun[G], acc[G][DPL];
#pragma unroll
      for (int h = 0; h < G; ++h) {
        mrun[h] = -INFINITY;
        lrun[h] = 0.f;
#pragma unroll
        for (int j = 0; j < DPL; ++j) acc[h][j] = 0.f;
      }
      (void)kn;
      (void)vn;
      const int newpos = a.T - 1;
      const int vidx = lane / LPV;
      const int my_i = vidx / G, my_h = vidx % G;
#pragma unroll 1
      for (int t = a.tile0; t < a.tile1; ++t) {
        const uint8_t* slot = wait_item();
        const int jn = newpos - t * kKvTilePos;
        if (jn >= 0 && jn < kKvTilePos) {  // (the same for all warps)
          uint16_t* kr = reinterpret_cast<uint16_t*>(const_cast<uint8_t*>(slot) + jn * row_bytes);
          uint16_t* vr = reinterpret_cast<uint16_t*>(const_cast<uint8_t*>(slot) + (kKvTilePos + jn) * row_bytes);
          if (!dead)
            for (int d = tid; d < HD; d += kConsumerWarps * 32) {
              kr[d] = f2bf(qkvn[G * HD + d]);
              vr[d] = f2bf(qkvn[(G + 1) * HD + d]);
            }
          cons_sync();
        }
        if (!dead) {
          const int p0 = t * kKvTilePos;
          const int npos = min(kKvTilePos, a.T - p0);
          float s[NV];
#pragma unroll
          for (int i = 0; i < PPW; ++i) {
            const int j = warp * PPW + i;
            float kf[DPL];
            if (j < npos) {
              const uint16_t* src = reinterpret_cast<const uint16_t*>(slot + j * row_bytes) + lane * DPL;
              if (DPL == 4) {
                const uint2 v = *reinterpret_cast<const uint2*>(src);
                kf[0] = bf16lo(v.x);
                kf[1] = bf16hi(v.x);
                kf[2 % DPL] = bf16lo(v.y);
                kf[3 % DPL] = bf16hi(v.y);
              } else {
                const uint32_t v = *reinterpret_cast<const uint32_t*>(src);
                kf[0] = bf16lo(v);
                kf[1 % DPL] = bf16hi(v);
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
          float sc_own = warp_transpose_reduce<NV>(s);
          if (warp * PPW + my_i >= npos) sc_own = -INFINITY;
          float bm = sc_own;
#pragma unroll
          for (int off = LPV * G; off < 32; off <<= 1) bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, off));
          float mnew[G], corr[G];
#pragma unroll
          for (int h = 0; h < G; ++h) {
            const float bmh = __shfl_sync(0xffffffffu, bm, h * LPV);
            mnew[h] = fmaxf(mrun[h], bmh);
            corr[h] = (mnew[h] == -INFINITY) ? 1.f : exp2f(mrun[h] - mnew[h]);
          }
          float mn_own = mnew[0];
#pragma unroll
          for (int h = 1; h < G; ++h)
            if (my_h == h) mn_own = mnew[h];
          const float pown = (sc_own == -INFINITY) ? 0.f : exp2f(sc_own - mn_own);
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
              const uint16_t* src = reinterpret_cast<const uint16_t*>(slot + (kKvTilePos + j) * row_bytes) + lane * DPL;
              float vf[DPL];
              if (DPL == 4) {
                const uint2 v = *reinterpret_cast<const uint2*>(src);
                vf[0] = bf16lo(v.x);
                vf[1] = bf16hi(v.x);
                vf[2 % DPL] = bf16lo(v.y);
                vf[3 % DPL] = bf16hi(v.y);
              } else {
                const uint32_t v = *reinterpret_cast<const uint32_t*>(src);
                vf[0] = bf16lo(v);
                vf[1 % DPL] = bf16hi(v);
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
      dead = cons_any(dead);  // (one verdict: the packing below is warp-collective)
      // the warps' states -> the unit's (max, sum, unnormalised output) per head
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
      constexpr int NPT = (G * HD + kConsumerWarps * 32 - 1) / (kConsumerWarps * 32);
      float ov[NPT], mv[NPT], lv[NPT];
#pragma unroll
      for (int i = 0; i < NPT; ++i) {
        const int idx = tid + i * kConsumerWarps * 32;
        ov[i] = mv[i] = lv[i] = 0.f;
        if (idx < G * HD) {
          const int h = idx / HD, d = idx % HD;
          float M = -INFINITY;
          for (int wi = 0; wi < kConsumerWarps; ++wi) M = fmaxf(M, wst[((size_t)wi * G + h) * (HD + 2) + HD]);
          float A = 0.f, Lsum = 0.f;
          if (M != -INFINITY) {
            for (int wi = 0; wi < kConsumerWarps; ++wi) {
              const float* r = wst + ((size_t)wi * G + h) * (HD + 2);
              const float e = exp2f(r[HD] - M);
              A = fmaf(e, r[d], A);
              Lsum = fmaf(e, r[HD + 1], Lsum);
            }
          }
          ov[i] = A;
          mv[i] = M;
          lv[i] = Lsum;
        }
      }
      cons_sync();  // (wst is overwritten below)
      if (w.nch == 1) {
        // the normalised output (bf16) of the group's heads, then their B blocks
        float* ob = red;
#pragma unroll
        for (int i = 0; i < NPT; ++i) {
          const int idx = tid + i * kConsumerWarps * 32;
          if (idx < G * HD) {
            const float wgt = (mv[i] == -INFINITY || !(lv[i] > 0.f)) ? 0.f : 1.f / lv[i];
            ob[idx] = bf16f(f2bf(wgt * ov[i]));
          }
        }
        cons_sync();
        if (warp < G * HD / kTileK && !dead) {
          const int kb = a.g * G * HD / kTileK + warp;
          float f[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) f[i] = ob[warp * kTileK + lane * 4 + i];
          pack4(w.pbo + (size_t)kb * PBS, w.exo + (size_t)kb * kWideMax + a.b, a.b, lane * 4, f);
        }
      } else if (!dead) {
        float* dst = w.attn_part + ((((size_t)a.b * p.hkv + a.g) * w.nch + a.c) * G) * (HD + 2);
#pragma unroll
        for (int i = 0; i < NPT; ++i) {
          const int idx = tid + i * kConsumerWarps * 32;
          if (idx < G * HD) {
            const int h = idx / HD, d = idx % HD;
            dst[(size_t)h * (HD + 2) + d] = ov[i];
            if (d == 0) {
              dst[(size_t)h * (HD + 2) + HD] = mv[i];
              dst[(size_t)h * (HD + 2) + HD + 1] = lv[i];
            }
          }
        }
      }
      cons_sync();
    }
  }

  // Chunk merge (more than one chunk per sequence and KV head): warp unit (token b, k block kb
  // of the attention output), four outputs per lane: per head, weights w_c = 2^(m_c - M) / L
  // with M = max_c m_c, L = sum_c 2^(m_c - M) l_c; output = sum_c w_c acc_c, in chunk order.
  __device__ void merge() {
    const size_t cst = (size_t)G * (HD + 2);
    const int nw = gridDim.x * kConsumerWarps;
#pragma unroll 1
    for (int wu = blockIdx.x * kConsumerWarps + warp; wu < p.B * p.kb_o && !dead; wu += nw) {
      const int b = wu / p.kb_o, kb = wu % p.kb_o;
      const int col = kb * kTileK + lane * 4;
      const int head = col / HD, d0 = col % HD;
      const int g = head / G, hl = head % G;
      const float* src = w.attn_part + (((size_t)b * p.hkv + g) * w.nch * G + hl) * (HD + 2);
      float mx = -INFINITY;
      for (int c = 0; c < w.nch; ++c) mx = fmaxf(mx, ldcg(src + c * cst + HD));
      float ls = 0.f;
      for (int c = 0; c < w.nch; ++c) {
        const float mc = ldcg(src + c * cst + HD);
        if (mc != -INFINITY) ls = fmaf(exp2f(mc - mx), ldcg(src + c * cst + HD + 1), ls);
      }
      float o[4] = {0.f, 0.f, 0.f, 0.f};
      for (int c = 0; c < w.nch; ++c) {
        const float mc = ldcg(src + c * cst + HD);
        const float wc = (mc == -INFINITY || !(ls > 0.f)) ? 0.f : exp2f(mc - mx) / ls;
        // (rows of hd + 2 floats: no vector loads)
#pragma unroll
        for (int i = 0; i < 4; ++i) o[i] = fmaf(wc, ldcg(src + c * cst + d0 + i), o[i]);
      }
      float f[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) f[i] = bf16f(f2bf(o[i]));
      pack4(w.pbo + (size_t)kb * PBS, w.exo + (size_t)kb * kWideMax + b, b, lane * 4, f);
    }
  }

  // ---- per-token phases (one CTA per token)

  __device__ const uint16_t* layer_in(int l, int t) const {
    if (l > 0) return w.xbuf + (size_t)t * p.d;
    if (p.tokens) return p.embed + (size_t)m->tok[t] * p.d;
    return p.hidden_in + (size_t)t * p.d;
  }

  // the first layer's input of every token, normalised, as B blocks
  __device__ void input_pack() {
    for (int t = blockIdx.x; t < p.B && !dead; t += gridDim.x) {
      const uint16_t* x = layer_in(0, t);
      uint4 v[MAXV];
#pragma unroll
      for (int j = 0; j < MAXV; ++j) {
        const int k = (tid + j * kConsumerWarps * 32) * 8;
        if (k < p.d) v[j] = ldcg4(x + k);
      }
      norm_pack(t, v, p.layers[0].attn_norm);
    }
  }

  // x_mid = bf16(x + output projection) of token t (summed from the projection's partials),
  // kept for the layer output; then bf16(rmsnorm(x_mid) * ffn_norm) as B blocks
  __device__ void xmid_pack(int l) {
    const WGeo go = wgeo(p, K_O, 0, gridDim.x);
    const size_t pst = (size_t)p.MB * kTileRows;
    for (int t = blockIdx.x; t < p.B && !dead; t += gridDim.x) {
      const uint16_t* x = layer_in(l, t);
      uint4 v[MAXV];
#pragma unroll
      for (int j = 0; j < MAXV; ++j) {
        const int k = (tid + j * kConsumerWarps * 32) * 8;
        if (k >= p.d) continue;
        v[j] = ldcg4(x + k);
        const int rb = k / kTileRows;
        const int nc = n_contrib(rb * go.kbs, go.kbs, go.T, gridDim.x);
        const float* src = p.part_o + ((size_t)rb * go.S * p.MB + t) * kTileRows + k % kTileRows;
        float o8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
        for (int c = 0; c < nc; ++c) {
          const float4 a0 = __ldcg(reinterpret_cast<const float4*>(src + (size_t)c * pst));
          const float4 a1 = __ldcg(reinterpret_cast<const float4*>(src + (size_t)c * pst + 4));
          o8[0] += a0.x; o8[1] += a0.y; o8[2] += a0.z; o8[3] += a0.w;
          o8[4] += a1.x; o8[5] += a1.y; o8[6] += a1.z; o8[7] += a1.w;
        }
        uint32_t* u = reinterpret_cast<uint32_t*>(&v[j]);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint16_t lo = f2bf(bf16lo(u[q]) + o8[2 * q]);
          const uint16_t hi = f2bf(bf16hi(u[q]) + o8[2 * q + 1]);
          u[q] = (uint32_t)lo | ((uint32_t)hi << 16);
        }
        *reinterpret_cast<uint4*>(w.xmid + (size_t)t * p.d + k) = v[j];
      }
      norm_pack(t, v, p.layers[l].ffn_norm);
    }
  }

  // Routing of token t from the router's partials: logits -> top-k by rank (ties to the lower
  // expert index, NaN as -inf) -> sigmoid scores normalised over the selection (summed in rank
  // order); written for the whole grid and for inspection.
  __device__ void route_tokens(int l) {
    const WGeo gr = wgeo(p, K_ROUTER, 0, gridDim.x);
    const size_t pst = (size_t)p.MB * kTileRows;
    float* lg = red;                                           // [kMaxExperts]
    int* selsm = reinterpret_cast<int*>(lg + kMaxExperts);     // [16]
    float* sg = reinterpret_cast<float*>(selsm + 16);          // [16]
    for (int t = blockIdx.x; t < p.B && !dead; t += gridDim.x) {
      if (tid < p.E) {
        const int rb = tid / kTileRows;
        const int nc = n_contrib(rb * gr.kbs, gr.kbs, gr.T, gridDim.x);
        const float* src = p.part_router + ((size_t)rb * gr.S * p.MB + t) * kTileRows + tid % kTileRows;
        float s = 0.f;
#pragma unroll 1
        for (int c0 = 0; c0 < nc; c0 += 8) {
          float v[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) v[j] = c0 + j < nc ? ldcg(src + (size_t)(c0 + j) * pst) : 0.f;
#pragma unroll
          for (int j = 0; j < 8; ++j) s += v[j];
        }
        lg[tid] = s;
        p.rt_logits[((size_t)l * p.rows + t) * p.E + tid] = s;
      }
      cons_sync();
      if (tid < p.E) {
        float v = lg[tid];
        if (v != v) v = -INFINITY;
        int rank = 0;
        for (int j = 0; j < p.E; ++j) {
          float x = lg[j];
          if (x != x) x = -INFINITY;
          rank += (x > v || (x == v && j < tid)) ? 1 : 0;
        }
        if (rank < p.topk) {
          selsm[rank] = tid;
          sg[rank] = 1.0f / (1.0f + expf(-v));
        }
      }
      cons_sync();
      if (warp == 0) {
        float ssum = 0.f;
        for (int k = 0; k < p.topk; ++k) ssum += sg[k];
        if (lane < p.topk) {
          const float gt = sg[lane] / ssum;
          w.sel[(size_t)t * p.topk + lane] = selsm[lane];
          w.selg[(size_t)t * p.topk + lane] = gt;
          p.rt_idx[((size_t)l * p.rows + t) * p.topk + lane] = selsm[lane];
          p.rt_topk_gate[((size_t)l * p.rows + t) * p.topk + lane] = gt;
        }
      }
      cons_sync();
    }
  }

  // Every CTA: the distinct experts of the step in ascending order (expert slots), each token's
  // selections as slots and gates, the tokens of each slot, and the (slot, token) pairs of the
  // SwiGLU phase (the shared expert: slot U, every token). Dense FFN: slot 0, every token.
  __device__ void local_routing() {
    int* mark = reinterpret_cast<int*>(red);  // [kMaxExperts]
    int* pairs = mark + kMaxExperts;          // [kWideMax * 17]
    const unsigned long long all = p.B >= 64 ? ~0ull : ((1ull << p.B) - 1ull);
    if (p.dense) {
      if (tid == 0) {
        m->U = 0;
        m->umask[0] = all;
        m->npairs = p.B;
      }
      for (int t = tid; t < p.B; t += kConsumerWarps * 32) pairs[t] = t;
      cons_sync();
      return;
    }
    for (int i = tid; i < kMaxExperts; i += kConsumerWarps * 32) mark[i] = 0;
    for (int i = tid; i <= kMaxExperts; i += kConsumerWarps * 32) m->umask[i] = 0ull;
    cons_sync();
    for (int i = tid; i < p.B * p.topk; i += kConsumerWarps * 32) mark[min(max(ldcg_i(w.sel + i), 0), p.E - 1)] = 1;
    cons_sync();
    if (warp == 0) {
      int U2 = 0;
      for (int j = 0; j < kMaxExperts / 32; ++j) {
        const int e = lane + 32 * j;
        const bool on = e < p.E && mark[e] != 0;
        const unsigned bal = __ballot_sync(0xffffffffu, on);
        const int rank = U2 + __popc(bal & ((1u << lane) - 1u));
        if (on) {
          mark[e] = rank + 1;
          m->elist[rank] = e;
        }
        U2 += __popc(bal);
      }
      if (lane == 0) m->U = min(U2, w.hmax - p.nsh);
    }
    cons_sync();
    const int U = m->U;
    for (int i = tid; i < p.B * p.topk; i += kConsumerWarps * 32) {
      const int t = i / p.topk, k = i % p.topk;
      const int u = min(mark[min(max(ldcg_i(w.sel + i), 0), p.E - 1)] - 1, U - 1);
      m->wsel[t][k] = (uint8_t)u;
      m->wgate[t][k] = ldcg(w.selg + i);
      atomicOr(&m->umask[u], 1ull << t);
      pairs[i] = (u << 8) | t;
    }
    if (p.nsh)
      for (int t = tid; t < p.B; t += kConsumerWarps * 32) pairs[p.B * p.topk + t] = (U << 8) | t;
    if (tid == 0) {
      if (p.nsh) m->umask[U] = all;
      m->npairs = p.B * p.topk + (p.nsh ? p.B : 0);
    }
    cons_sync();
    if (tid == 0) mbar_arrive(&m->rt_bar);  // the producer and the MMA warp may take the routed experts
  }
  __device__ __forceinline__ static int ldcg_i(const int32_t* a) { return __ldcg(a); }

  // SwiGLU of every (expert slot, token) pair, one warp per pair and k block of h: h =
  // bf16(silu(gate) * up) from the gate/up partials (each row block: 64 gate rows, then the
  // matching 64 up rows), as B blocks of the slot's down projection.
  __device__ void swiglu_pack(int U) {
    const int* pairs = reinterpret_cast<const int*>(red) + kMaxExperts;
    const WGeo gr = wgeo(p, K_RTGU, U, gridDim.x), gs = wgeo(p, K_SHGU, 0, gridDim.x);
    const size_t pst = (size_t)p.MB * kTileRows;
    const int nw = gridDim.x * kConsumerWarps;
    const int nu = m->npairs * p.kb_i;
#pragma unroll 1
    for (int wu = blockIdx.x * kConsumerWarps + warp; wu < nu && !dead; wu += nw) {
      const int pi = wu / p.kb_i, kb = wu % p.kb_i;
      const int pr = pairs[pi];
      const int u = pr >> 8, t = pr & 255;
      const bool sh = u >= U;
      const int j0 = kb * kTileK + lane * 4;
      const int rbg = j0 / 64, r = j0 % 64;
      const WGeo& g = sh ? gs : gr;
      const int seg = sh ? rbg : u * p.n_rb_gu + rbg;
      const int nc = n_contrib(seg * g.kbs, g.kbs, g.T, gridDim.x);
      const float* src = (sh ? p.part_shgu : p.part_rtgu) + ((size_t)seg * g.S * p.MB + t) * kTileRows;
      float gv[4] = {0.f, 0.f, 0.f, 0.f}, uv[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
      for (int c = 0; c < nc; ++c) {
        const float4 a = __ldcg(reinterpret_cast<const float4*>(src + (size_t)c * pst + r));
        const float4 b = __ldcg(reinterpret_cast<const float4*>(src + (size_t)c * pst + 64 + r));
        gv[0] += a.x; gv[1] += a.y; gv[2] += a.z; gv[3] += a.w;
        uv[0] += b.x; uv[1] += b.y; uv[2] += b.z; uv[3] += b.w;
      }
      float f[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) f[i] = bf16f(f2bf((gv[i] / (1.0f + expf(-gv[i]))) * uv[i]));
      const size_t blk = (size_t)u * p.kb_i + kb;
      pack4(w.pbh + blk * PBS, w.exh + blk * kWideMax + t, t, lane * 4, f);
    }
  }

  // Layer output of token t: x_mid + the down partials of its routed slots (gate-weighted
  // already) and of the shared expert, rounded to bf16; then the next layer's (or the final)
  // RMSNorm as B blocks.
  __device__ void layer_out(int l, int U) {
    const WGeo gd = wgeo(p, K_D, U, gridDim.x);
    const size_t pst = (size_t)p.MB * kTileRows;
    const int nsel = p.dense ? 0 : p.topk;
    for (int t = blockIdx.x; t < p.B && !dead; t += gridDim.x) {
      uint4 v[MAXV];
#pragma unroll
      for (int j = 0; j < MAXV; ++j) {
        const int k = (tid + j * kConsumerWarps * 32) * 8;
        if (k >= p.d) continue;
        v[j] = ldcg4(w.xmid + (size_t)t * p.d + k);
        const int rb = k / kTileRows;
        float y[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
        for (int s = 0; s < nsel + p.nsh; ++s) {
          const int u = s < nsel ? (int)m->wsel[t][s] : U;
          const int seg = u * p.n_rb_d + rb;
          const int nc = n_contrib(seg * gd.kbs, gd.kbs, gd.T, gridDim.x);
          const float* src = p.part_d + ((size_t)seg * gd.S * p.MB + t) * kTileRows + k % kTileRows;
#pragma unroll 1
          for (int c = 0; c < nc; ++c) {
            const float4 a0 = __ldcg(reinterpret_cast<const float4*>(src + (size_t)c * pst));
            const float4 a1 = __ldcg(reinterpret_cast<const float4*>(src + (size_t)c * pst + 4));
            y[0] += a0.x; y[1] += a0.y; y[2] += a0.z; y[3] += a0.w;
            y[4] += a1.x; y[5] += a1.y; y[6] += a1.z; y[7] += a1.w;
          }
        }
        uint32_t* u32 = reinterpret_cast<uint32_t*>(&v[j]);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint16_t lo = f2bf(bf16lo(u32[q]) + y[2 * q]);
          const uint16_t hi = f2bf(bf16hi(u32[q]) + y[2 * q + 1]);
          u32[q] = (uint32_t)lo | ((uint32_t)hi << 16);
        }
        *reinterpret_cast<uint4*>(w.xbuf + (size_t)t * p.d + k) = v[j];
        if (l == p.L - 1 && p.hidden_out) *reinterpret_cast<uint4*>(p.hidden_out + (size_t)t * p.d + k) = v[j];
      }
      if (l + 1 < p.L) norm_pack(t, v, p.layers[l + 1].attn_norm);
      else if (p.V > 0) norm_pack(t, v, p.final_norm);
    }
  }

  // LM head row block rb: the logits of every token (summed from the partials) and each token's
  // largest logit of the block (ties to the lower row) folded into amax[t].
  __device__ void lm_final() {
    const WGeo g = wgeo(p, K_LM, 0, gridDim.x);
    const size_t pst = (size_t)p.MB * kTileRows;
    float* out = p.logits ? p.logits : p.logits_ws;
    for (int rb = blockIdx.x; rb < p.n_rb_lm && !dead; rb += gridDim.x) {
      const int nc = n_contrib(rb * g.kbs, g.kbs, g.T, gridDim.x);
      for (int t = warp; t < p.B; t += kConsumerWarps) {
        const float* src = p.part_lm + ((size_t)rb * g.S * p.MB + t) * kTileRows;
        float bv = -INFINITY;
        int bi = lane;
#pragma unroll
        for (int jj = 0; jj < kTileRows / 32; ++jj) {
          const int i = lane + 32 * jj, r = rb * kTileRows + i;
          float v = -INFINITY;
          if (r < p.V) {
            v = 0.f;
            for (int c = 0; c < nc; ++c) v += ldcg(src + (size_t)c * pst + i);
            out[(size_t)t * p.V + r] = v;
          }
          if (jj == 0 || v > bv) {
            bv = v;
            bi = i;
          }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
          const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
          const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
          if (ov > bv || (ov == bv && oi < bi)) {
            bv = ov;
            bi = oi;
          }
        }
        if (lane == 0)
          atomicMax(p.amax + t, ((unsigned long long)float_key(bv) << 32) |
                                    (unsigned long long)(0xFFFFFFFFu - (unsigned)(rb * kTileRows + bi)));
      }
    }
  }

  // ---- the step

  __device__ void stamp_layer(int l) {
    if (blockIdx.x == 0 && tid == 0) p.layer_ts[l] = gtimer();
  }

  __device__ void run() {
    if (warp == 0) tmem_alloc(&m->tmem_base, kTmemCols);
    tc_fence_before();
    cons_sync();
    tc_fence_after();
    tmem = m->tmem_base;
    if (tid == 0) mbar_arrive(&m->tm_ready);
    input_pack();
    gbar();
#pragma unroll 1
    for (int l = 0; l < p.L; ++l) {
      stamp_layer(l);
      gemv(K_QKV, 0);
      gbar();
      attention(l);
      gbar();
      if (w.nch > 1) merge();
      gbar();
      gemv(K_O, 0);
      gbar();
      xmid_pack(l);
      gbar();
      if (!p.dense) gemv(K_ROUTER, 0);
      if (p.dense || p.nsh) gemv(K_SHGU, 0);
      gbar();
      if (!p.dense) route_tokens(l);
      gbar();
      local_routing();
      const int U = m->U;
      if (!p.dense) gemv(K_RTGU, U);
      gbar();
      swiglu_pack(U);
      gbar();
      gemv(K_D, U);
      gbar();
      layer_out(l, U);
      gbar();
    }
    stamp_layer(p.L);
    if (p.V > 0) {
      gemv(K_LM, 0);
      gbar();
      lm_final();
      gbar();
      if (blockIdx.x == 0 && tid < p.B && !dead) {
        const unsigned long long key = atomicExch(p.amax + tid, 0ull);
        if (p.next_tokens) p.next_tokens[tid] = (int)(0xFFFFFFFFu - (unsigned)(key & 0xFFFFFFFFull));
      }
    }
    if (blockIdx.x == 0 && tid < p.B && !dead) p.lengths[p.seq0 + tid] = m->len[tid] + 1;
    if (blockIdx.x == 0 && tid == 0) p.layer_ts[p.L + 1] = gtimer();
    // TMEM is freed once the MMA warp has finished (bounded wait)
    if (warp == 0) {
      if (lane == 0) {
        const unsigned long long t0 = gtimer();
        while (!mbar_try_wait(&m->mma_done, 0) && gtimer() - t0 < p.timeout_ns) {
        }
      }
      __syncwarp();
      tc_fence_after();
      tmem_free(tmem, kTmemCols);
    }
  }
};

// ---------------------------------------------------------------------------------------------

template <int NR, int HD, int G>
__global__ void __launch_bounds__(kThreads, 1)
    wide_step_kernel(const __grid_constant__ KParams p, const __grid_constant__ WideParams w) {
  extern __shared__ __align__(128) uint8_t smem[];
  const WLayout L = wlayout(p.ring, NR, HD, G);
  uint8_t* ring = smem + L.ring_off;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.full_off);
  uint64_t* empty = reinterpret_cast<uint64_t*>(smem + L.empty_off);
  uint64_t* mempty = reinterpret_cast<uint64_t*>(smem + L.mempty_off);
  float* red = reinterpret_cast<float*>(smem + L.red_off);
  WMisc* m = reinterpret_cast<WMisc*>(smem + L.misc_off);
  const int tid = threadIdx.x;
  if (tid == 0) {
    for (int s = 0; s < p.ring; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
      mbar_init(&mempty[s], 1);
    }
    mbar_init(&m->rt_bar, 1);
    mbar_init(&m->mma_done, 1);
    mbar_init(&m->tm_ready, 1);
    m->stages_begun = 0;
    for (int i = 0; i < kNGW; ++i) {
      mbar_init(&m->tfull[i], 2);  // MMA commit + the MMA thread's release of the block scales
      mbar_init(&m->tempty[i], kConsumerWarps);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (tid < kWideMax) {
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
      WProducer<NR, HD, G> prod(p, w, ring, full, empty, mempty, m);
      prod.run();
    } else if (tid == (kConsumerWarps + 1) * 32) {
      WMma<NR, HD, G> mma(p, w, ring, full, mempty, m);
      mma.run();
    }
    return;
  }
  WConsumer<NR, HD, G> cons(p, w, ring, full, empty, red, m);
  cons.run();
}

}  // namespace wide
}  // namespace dec
