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
//               synchronisation wait).
//   warps 0..7  consumers: hand each weight tile to the tensor cores (thread 0 issues
//               tcgen05.mma on the raw E4M3 tile and the activations split into E4M3 pieces,
//               accumulating in TMEM), add the tiles' products into fp32 registers with their
//               block scales, and publish split-K partial sums with a releasing counter arrival
//               (no CTA ever waits for the result of its own arrival); attention runs on the
//               CUDA cores.
// Cross-CTA data flow of a layer: the q/k/v, output-projection and router partials are read
// directly by every CTA that needs them (attention units, the x_mid norm, the routing, which
// every CTA computes itself); the attention chunks of a (sequence, KV head) are merged in slices
// by all of its chunks' CTAs; SwiGLU rows and the layer output row blocks are finalised by CTAs
// designated per group (spread evenly over the grid), which wait for the group's counter and
// publish a counter arrival (SwiGLU) or an epoch flag (layer output). There is no grid barrier:
// each consumer waits only for the data it reads. Every wait is bounded and turns into an error
// status instead of a hang. Weight copies carry an L2 evict-first hint, so the streamed weights
// do not evict the small exchange data the hops read back.
#pragma once
#include "dec_prims.cuh"

namespace dec {

// ---------------------------------------------------------------------------------------------
// shared-memory layout (identical on host and device)

struct SmemLayout {
  int ring_off, full_off, empty_off, mempty_off, xs_off, red_off, misc_off, total;
};

constexpr int kMaxExperts = 128;
// Tensor-core tiles: every tile's product gets its own kMmaN-column TMEM slice; tiles are handed
// to the consumers in groups of up to kGT (consecutive tiles of one segment), kNG groups in
// flight (all 512 TMEM columns), so the consumers synchronise with the MMA warp once per group.
// Activation k blocks per stage at most kMaxKb.
constexpr int kMmaN = 16;
constexpr int kGT = 8;
constexpr int kNG = 4;
constexpr int kTmemCols = kNG * kGT * kMmaN;  // 512
constexpr int kMaxKb = 64;
constexpr int kMaxRing = 16;

// Layout of the B operand (a stage's activations as E4M3 pieces, the canonical K-major layout
// of 8-row x 16-byte core matrices) for a step of B tokens: each k block of 128 activations
// takes rpad rows (2B: rows 2b, 2b + 1 are token b's two pieces; 3 tokens pad to 8, 5..8 to 16),
// and pk consecutive k blocks share one block of nrb rows (8, or 16 for B > 4), whose MMA (N = 16)
// yields their columns side by side. With nrb = 8 the second 8-row group of N aliases the first.
struct BGeo {
  int rpad, pk, nrb;
};
__host__ __device__ inline BGeo bgeo(int B) {
  BGeo g;
  g.rpad = B <= 1 ? 2 : B <= 2 ? 4 : B <= 4 ? 8 : 16;
  g.nrb = g.rpad <= 8 ? 8 : 16;
  g.pk = g.rpad <= 8 ? 8 / g.rpad : 1;
  return g;
}
constexpr int kProducerTrace = 128;  // trace words reserved for CTA 0's producer

constexpr int kWaitMax = 128;  // conditions one CTA-wide wait table holds
constexpr int kDRowMajorMax = 12;  // down projections of at most this many expert slots: row-block major
constexpr int kListCap = 1024;     // contributor slots one down-projection row block may gather
// The consumer thread that publishes a CTA's results (releasing arrivals and flags, preceded by
// a CTA barrier) and resets the counters it finalised: a thread of the last warp, so that warp 0,
// which polls in every CTA-wide wait, does not stall on the release.
constexpr int kPubThread = (kConsumerWarps - 1) * 32;

struct Misc {
  const unsigned* wt_addr[kWaitMax];  // CTA-wide wait: *wt_addr[i] >= wt_want[i] for all i
  unsigned wt_want[kWaitMax];
  uint64_t rt_bar;  // consumers -> producer: this layer's routing is in elist / U (one phase per layer)
  int flag;
  int nfin;
  int U;
  int len[kMaxBatch];
  int elist[kMaxExperts];
  float gate[kMaxBatch][kMaxExperts + 1];
  float rsum[kConsumerWarps][kMaxBatch];
  int tok[kMaxBatch];
  // tensor-core tiles: the scale exponent a of each token's staged k block (its pieces encode
  // x * 2^a), the count of GEMV stages whose operand the consumers have staged (consumers -> MMA
  // warp; a count, so that two stages staged before the MMA warp looks cannot be mistaken for
  // one), the MMA warp's "done" barrier, per group of TMEM slices a "products ready" (MMA commit)
  // and a "products read" (one arrival per consumer warp) barrier, and the TMEM base address
  int8_t xexp[kMaxBatch][kMaxKb];
  unsigned stages_staged;
  uint64_t mma_done;
  uint64_t tfull[kNG], tempty[kNG];
  float2 hdr[kNG][kGT];  // the block scales of each group's tiles (their slots may be refilled first)
  uint32_t tmem_base;
};

struct WaitCond {
  const unsigned* addr;  // null: holds at once
  unsigned want;         // holds once *addr >= want
};

__host__ __device__ inline int align_up(int x, int a) { return (x + a - 1) / a * a; }

__host__ __device__ inline SmemLayout smem_layout(int ring, int bm, int xmax, int hd, int group) {
  SmemLayout s;
  s.ring_off = 0;
  s.full_off = align_up(ring * kSlotBytes, 128);
  s.empty_off = s.full_off + ring * 8;
  s.mempty_off = s.empty_off + ring * 8;  // a slot's tiles read by the tensor cores (MMA commit)
  s.xs_off = align_up(s.mempty_off + ring * 8, 128);
  // the stage's activations as tensor-core B operand blocks, for any step batch up to bm
  int xs_bytes = 0;
  for (int b = 1; b <= bm; ++b) {
    const BGeo g = bgeo(b);
    const int bytes = (xmax / 128 + g.pk - 1) / g.pk * g.nrb * 128;
    xs_bytes = bytes > xs_bytes ? bytes : xs_bytes;
  }
  s.red_off = align_up(s.xs_off + xs_bytes, 128);
  int red_gemv = 2 * kTileRows * bm * 4;
  // attention: the warps' states, or the unit's q/k/v (+ raw sums) and, in multi-position steps,
  // every new token's key and value
  int red_attn = kConsumerWarps * group * (hd + 2) * 4;
  const int red_qkv = (2 * (group + 2) * hd + 2 * bm * hd) * 4;
  red_attn = red_attn > red_qkv ? red_attn : red_qkv;
  int red_fin = (bm * kTileRows + kListCap + 16) * 4;
  int red = red_gemv > red_attn ? red_gemv : red_attn;
  red = red > red_fin ? red : red_fin;
  s.misc_off = align_up(s.red_off + red, 128);
  s.total = align_up(s.misc_off + (int)sizeof(Misc), 128);
  return s;
}

// GEMV stage kinds
enum Kind : int { K_QKV = 0, K_O, K_ROUTER, K_SHGU, K_RTGU, K_D, K_LM };

// per-CTA dependency stamps of a layer (trace words from kTraceSlots on)
enum Stamp : int {
  S_QKV_TILES = 0,  // q/k/v tiles consumed
  S_QKV_DONE,       // q/k/v partials published
  S_ATTN_DONE,      // the CTA's attention units merged
  S_OGRP_READY,     // the attention outputs its projection tiles read are final
  S_O_TILES,        // output-projection tiles consumed
  S_O_DONE,         // output-projection partials published
  S_XMID_READY,     // x_mid summed and normalised
  S_FFN_PRE_DONE,   // router partials published
  S_ROUTED,         // routing known
  S_GU_TILES,       // routed (or dense) gate/up tiles consumed
  S_GU_DONE,        // gate/up partials published, SwiGLU finalisers run
  S_H_READY,        // the SwiGLU rows its down tiles read are final
  S_D_TILES,        // down-projection tiles consumed
  S_D_DONE,         // down partials published, finalisers run
  S_BARRIER,        // layer done (its down stage and finalisers)
};

// ---------------------------------------------------------------------------------------------
// schedule arithmetic shared by producer and consumers

// 32-bit arithmetic: a stage has far fewer than 2^31 / grid tiles (the host checks the largest)
__device__ __forceinline__ int range_lo(int T, int c, int G) { return (int)((unsigned)T * (unsigned)c / (unsigned)G); }
__device__ __forceinline__ int owner_of(int t, int T, int G) {
  return (int)(((unsigned)(t + 1) * (unsigned)G - 1u) / (unsigned)T);
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
  int kbs;  // tiles per segment (the k blocks one output row block sums)
  int tpe;  // expert stages: tiles of one expert in a row (one run)
  int rbm;  // down projections: row-block major (else expert major)
};

__device__ __forceinline__ StageGeo stage_geo(const KParams& p, int kind, int U) {
  StageGeo g;
  g.tpe = 0;
  g.rbm = 0;
  switch (kind) {
    case K_QKV: g.kbs = p.kb_d; g.T = p.n_rb_qkv * p.kb_d; break;
    case K_O: g.kbs = p.kb_o; g.T = p.n_rb_d * p.kb_o; break;
    case K_ROUTER: g.kbs = p.kb_d; g.T = p.n_rb_router * p.kb_d; break;
    case K_SHGU: g.kbs = p.kb_d; g.T = p.n_rb_gu * p.kb_d; break;
    case K_RTGU: g.kbs = p.kb_d; g.tpe = p.n_rb_gu * p.kb_d; g.T = U * g.tpe; break;
    // Down projections of the nv = U + nsh active expert slots (routed, then the shared one).
    // Few slots: row-block major, segment rb = the kb_i k blocks of row block rb of every slot in
    // turn, so one output row block's tiles are contiguous and split among few CTAs. Many slots
    // (large batches): expert major, one expert's row blocks after another (segments of kb_i),
    // so a CTA's range spans few experts (whose SwiGLU rows it stages).
    case K_D: {
      const int nv = U + p.nsh;
      g.rbm = nv <= kDRowMajorMax;
      g.tpe = g.rbm ? p.kb_i : p.n_rb_d * p.kb_i;
      g.kbs = g.rbm ? nv * p.kb_i : p.kb_i;
      g.T = p.n_rb_d * nv * p.kb_i;
      break;
    }
    default: g.kbs = p.kb_d; g.T = p.n_rb_lm * p.kb_d; break;
  }
  return g;
}

// Walks a stage's tiles in order (no divisions per tile). Plain stages are one contiguous run of
// tiles; the routed gate/up stage is a run of tpe tiles per expert slot u, at that expert's
// weights; the down stage is, per output row block rb, a run of kb_i tiles of each expert slot u
// (the shared expert after the routed ones), at row block rb of that expert's weights.
struct TileCursor {
  const uint8_t* addr;
  int u, r, rb;  // expert stages: expert slot, tile within its run, (down) output row block
  __device__ __forceinline__ static const uint8_t* expert_base(const KParams& p, const LayerDev& Ld, int kind, int u,
                                                               int U, const int* elist) {
    if (kind == K_RTGU) return Ld.e_gu + (size_t)elist[u] * p.e_gu_stride;
    return u < U ? Ld.e_d + (size_t)elist[u] * p.e_d_stride : Ld.sh_d;
  }
  __device__ void init(const KParams& p, const LayerDev& Ld, int kind, int t, const StageGeo& g, int U,
                       const int* elist) {
    if (kind == K_RTGU || (kind == K_D && !g.rbm)) {
      u = t / g.tpe;
      r = t - u * g.tpe;
      addr = expert_base(p, Ld, kind, u, U, elist) + (size_t)r * kTileBytes;
      return;
    }
    if (kind == K_D) {
      rb = t / g.kbs;
      const int k = t - rb * g.kbs;
      u = k / g.tpe;
      r = k - u * g.tpe;
      addr = expert_base(p, Ld, kind, u, U, elist) + ((size_t)rb * g.tpe + r) * kTileBytes;
      return;
    }
    const uint8_t* base = kind == K_QKV ? Ld.qkv
                        : kind == K_O ? Ld.o
                        : kind == K_ROUTER ? Ld.router
                        : kind == K_SHGU ? Ld.sh_gu
                                         : p.lm;
    u = 0;
    r = t;
    addr = base + (size_t)t * kTileBytes;
  }
  // advance to the next tile; past the stage's last expert there is none (the caller stops first)
  __device__ __forceinline__ void next(const KParams& p, const LayerDev& Ld, int kind, const StageGeo& g, int U,
                                       const int* elist) {
    addr += kTileBytes;
    if ((kind == K_RTGU || (kind == K_D && !g.rbm)) && ++r == g.tpe) {
      r = 0;
      ++u;
      if (u * g.tpe < g.T) addr = expert_base(p, Ld, kind, u, U, elist);
    }
    if (kind == K_D && g.rbm && ++r == g.tpe) {
      r = 0;
      if (++u * g.tpe == g.kbs) {
        u = 0;
        ++rb;
      }
      if (rb < p.n_rb_d) addr = expert_base(p, Ld, kind, u, U, elist) + (size_t)rb * g.tpe * kTileBytes;
    }
  }
};

// Position of a GEMV stage's tile, advanced without divisions (consumers and the MMA warp walk
// the same sequence): segment, k block within it, and for the down projection the expert slot v,
// the k block kx within the expert's run and the run's place xj among the staged SwiGLU rows.
struct TilePos {
  int seg, kb, kx, v, rv, xj;
  __device__ void init(const KParams& p, const StageGeo& g, int kind, int t0, int t1) {
    seg = kb = kx = v = rv = xj = 0;
    if (t1 <= t0) return;
    seg = t0 / g.kbs;
    kb = t0 - seg * g.kbs;
    kx = kb;
    if (kind == K_D) {
      v = g.rbm ? kb / g.tpe : t0 / g.tpe;          // expert slot of the first tile
      rv = g.rbm ? kb - v * g.tpe : t0 - v * g.tpe;  // its place in that expert's run
      kx = rv % p.kb_i;                              // and in its k-block sweep
    }
  }
  __device__ __forceinline__ void next(const KParams& p, const StageGeo& g, int kind, int nv) {
    if (++kb == g.kbs) {
      kb = 0;
      ++seg;
    }
    if (kind != K_D) {
      kx = kb;
    } else {
      if (++kx == p.kb_i) kx = 0;
      if (++rv == g.tpe) {
        rv = 0;
        if (++v == nv) v = 0;
        if (++xj == nv) xj = 0;
      }
    }
  }
  // k block of the staged activations the tile multiplies
  __device__ __forceinline__ int kbi(const KParams& p, int kind) const { return kind == K_D ? xj * p.kb_i + kx : kx; }
};

// attention work units: (sequence b, KV head g, context chunk c)
struct AttnUnit {
  int b, g, c, tile0, tile1, T;
};
__device__ __forceinline__ AttnUnit attn_unit(const KParams& p, const Misc* m, int u, int soff) {
  AttnUnit a;
  int per_b = p.hkv * p.nch;
  a.b = u / per_b;
  a.g = (u / p.nch) % p.hkv;
  a.c = u % p.nch;
  a.T = m->len[a.b] + soff + 1;  // (m->len: lengths at the launch; soff: resident steps done)
  int ntile = (a.T + kKvTilePos - 1) / kKvTilePos;
  int tpc = (ntile + p.nch - 1) / p.nch;
  a.tile0 = min(ntile, a.c * tpc);
  a.tile1 = min(ntile, a.tile0 + tpc);
  return a;
}

__device__ __forceinline__ size_t kv_row(const KParams& p, int l, int b, int g, int pos) {
  const int slot = p.mpos ? p.seq0 : p.seq0 + b;  // (consecutive positions share one slot)
  return ((((size_t)l * p.slots + slot) * p.hkv + g) * p.max_ctx + pos) * p.hd;
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
  unsigned item = 0;  // slots issued so far in this step
  int pslot = 0;      // ring slot of the next item (item % ring, kept without divisions)
  unsigned plap = 0;  // times the ring has wrapped (item / ring)
  // L2 eviction policies of the bulk copies. Weight tiles: evict first. They are read once per
  // step (~1.9 GB go through L2 per step at the 8-layer stack); without the hint they push out
  // the small exchange data (partial sums, counters, activations) that the CTAs' hops read back
  // from L2, and the step is ~4% longer. KV rows: normal priority (measured marginally better).
  uint64_t pol_stream = 0, pol_kv = 0;
  unsigned landed = 0;  // issued slots seen to have landed, in issue order
  int lslot = 0;        // ring slot of item `landed`
  unsigned llap = 0;    // its lap (landed / ring)
  bool dead = false;
  int stamp = 0;
  int soff = 0;       // resident steps done in this launch
  unsigned lay = 0;   // layers done in this launch (the routing barrier's phase)

  // CTA 0's producer records (code, %globaltimer) pairs in the last kProducerTrace words:
  // code = what << 4 | event, event 0 = first copy of a stage issued, 1 = last copy issued
  // (what: GEMV kind, 7 attention, 9 routing wait with 0 = begin, 1 = flag seen).
  __device__ void trace(int code) {
    if (DEC_TRACE && blockIdx.x == 0 && stamp + 1 < kProducerTrace) {
      p.trace[kTraceSlots - kProducerTrace + stamp] = (unsigned long long)code;
      p.trace[kTraceSlots - kProducerTrace + stamp + 1] = gtimer();
      stamp += 2;
    }
  }

  // Slots are released by the consumer warps (count kConsumerWarps on `empty`), or, for weight
  // tiles of the tensor-core kernels, by the MMA warp's commit once the MMAs reading them are
  // done (count 1 on `mempty`). One bit per slot (ring <= kMaxRing <= 32): whether its last use
  // completes `mempty`, and the parity of the number of uses of each kind so far.
  uint64_t* mempty;
  uint32_t last_mma = 0, ne_par = 0, nm_par = 0;

  __device__ Producer(const KParams& p_, uint8_t* r, uint64_t* f, uint64_t* e, uint64_t* me, Misc* m_)
      : p(p_), ring(r), full(f), empty(e), m(m_), mempty(me) {}

  // every bulk copy source must lie inside its allocation (checked before the copy is issued)
  __device__ __forceinline__ static bool within(const void* src, size_t bytes, const void* base, size_t extent) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(src), b = reinterpret_cast<uintptr_t>(base);
    return a >= b && a + bytes <= b + extent && (a & 15u) == 0 && (bytes & 15u) == 0;
  }

  // claim the next slot: wait until at most p.inflight - 1 of the CTA's copies are still in
  // flight, then until the consumers released the slot.
  // The cap matters when a stage starts: every CTA finds several free slots at the same moment,
  // and the memory system serves all the copies it is handed interleaved, so a whole ring's
  // worth from every CTA would make even each CTA's first slot land only when nearly all of it
  // has. With a few copies per CTA in flight (enough to keep the memory busy), the first slots
  // land after about one unloaded latency and the rest follow at the rate they are consumed.
  // (p.inflight <= ring: the slot of item `landed` is never re-armed before it is checked.)
  __device__ bool claim(int& slot, bool mma_use) {
    while (item - landed >= (unsigned)p.inflight) {
      if (!mbar_wait(&full[lslot], llap & 1, p, 12)) {
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
      // the previous use's phase: the (count - 1)-th completion, parity = count's parity flipped
      const bool pm = (last_mma & bit) != 0;
      const unsigned par = (((pm ? nm_par : ne_par) >> slot) & 1u) ^ 1u;
      if (!mbar_wait(pm ? &mempty[slot] : &empty[slot], par, p, 10)) {
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

  __device__ void issue_gemv(int kind, int l, int U, const int* elist) {
    if (dead) return;
    const StageGeo g = stage_geo(p, kind, U);
    const int G_ = gridDim.x;
    const int t0 = range_lo(g.T, blockIdx.x, G_), t1 = range_lo(g.T, blockIdx.x + 1, G_);
    const LayerDev& Ld = p.layers[l < p.L ? l : 0];
    if (t1 > t0) trace(kind << 4);
    // a slot takes the next kSlotTiles tiles of the CTA's range (fewer at its end): one copy when
    // they are adjacent in memory, one per tile otherwise (an expert boundary). The tile address
    // is advanced tile by tile (no divisions in the loop).
    TileCursor cur;
    if (t1 > t0) cur.init(p, Ld, kind, t0, g, U, elist);
    for (int t = t0; t < t1; t += kSlotTiles) {
      int slot;
      if (!claim(slot, BM >= 2)) return;  // (tensor-core kernels: the MMA warp frees weight slots)
      const int n = min(kSlotTiles, t1 - t);
      const uint8_t* src[kSlotTiles];
      bool ok = true;
#pragma unroll
      for (int j = 0; j < kSlotTiles; ++j) {
        src[j] = cur.addr;
        if (j < n) {
          ok = ok && within(src[j], kTileBytes, p.warena, p.warena_bytes);
          cur.next(p, Ld, kind, g, U, elist);
        }
      }
      uint8_t* dst = ring + (size_t)slot * kSlotBytes;
      if (!ok) {
        raise_err(p, kDevBadArg, 30);
        mbar_arrive(&full[slot]);  // keep the ring consistent; the status word stops the step
        advance();
        continue;
      }
      mbar_arrive_expect_tx(&full[slot], (unsigned)n * kTileBytes);
      if (n == 2 && src[1] == src[0] + kTileBytes) {
        bulk_g2s_hint(dst, src[0], 2 * kTileBytes, &full[slot], pol_stream);
      } else {
        for (int j = 0; j < n; ++j)
          bulk_g2s_hint(dst + (size_t)j * kTileBytes, src[j], kTileBytes, &full[slot], pol_stream);
      }
      advance();
    }
    if (t1 > t0) trace(kind << 4 | 1);
  }

  __device__ void issue_attn(int l) {
    if (dead) return;
    if (soff > 0) {
      // Resident steps: the KV cache is not static data. The previous step's keys and values
      // (written by whichever CTA held their position) must be in place before this step's KV
      // tiles are copied, and the producer may otherwise run steps ahead of them: wait (bounded)
      // for the previous step's token flag, published after all of that step's work, then order
      // the copies (async proxy) after the writes it made visible.
      const unsigned want = p.epoch + (unsigned)soff - 1u;
      const unsigned long long t0 = gtimer();
      for (unsigned it = 1; ld_acquire(p.tok_flag) < want; ++it) {
        if ((it & 15u) == 0) {
          if (aborted(p)) {
            dead = true;
            return;
          }
          if (gtimer() - t0 > p.timeout_ns) {
            raise_err(p, kDevTimeout, 32);
            dead = true;
            return;
          }
        }
      }
      fence_proxy_async_global();
    }
    const int NU = p.B * p.hkv * p.nch;
    const unsigned row_bytes = HD * 2;
    for (int u = blockIdx.x; u < NU; u += gridDim.x) {
      AttnUnit a = attn_unit(p, m, u, soff);
      for (int t = a.tile0; t < a.tile1; ++t) {
        int slot;
        if (!claim(slot, false)) return;
        int p0 = t * kKvTilePos;
        int n = min(kKvTilePos, a.T - p0);
        uint8_t* dst = ring + (size_t)slot * kSlotBytes;
        const size_t r0 = kv_row(p, l, a.b, a.g, p0);
        if (n < 1 || n > kKvTilePos || !within(p.kc + r0, n * row_bytes, p.kc, p.kv_bytes) ||
            !within(p.vc + r0, n * row_bytes, p.vc, p.kv_bytes)) {
          raise_err(p, kDevBadArg, 31);
          mbar_arrive(&full[slot]);
          advance();
          continue;
        }
        mbar_arrive_expect_tx(&full[slot], 2u * n * row_bytes);
        bulk_g2s_hint(dst, p.kc + r0, n * row_bytes, &full[slot], pol_kv);
        bulk_g2s_hint(dst + kKvTilePos * row_bytes, p.vc + r0, n * row_bytes, &full[slot], pol_kv);
        advance();
      }
    }
  }

  // Routed experts are known only after the router: the CTA's consumers compute the routing and
  // arrive on the routing mbarrier (one phase per layer) once it is in shared memory.
  __device__ bool routing(int l, int& U, int* elist) {
    if (dead) return false;
    trace(9 << 4);
    if (!mbar_wait(&m->rt_bar, lay & 1u, p, 11)) {
      dead = true;
      return false;
    }
    trace(9 << 4 | 1);
    U = min(max(m->U, 0), p.umax);
    for (int i = 0; i < U; ++i) elist[i] = min(max(m->elist[i], 0), p.E - 1);
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

  // The load program: per layer q/k/v, KV tiles, output projection, router, shared expert,
  // (routing) routed gate/up, down; then the LM head. Every GEMV stage goes through the one
  // issue_gemv call below, so its code exists once in the kernel.
  __device__ void run() {
    int elist[kMaxExperts];
    int U = 0;
    pol_stream = l2_policy(true);
    pol_kv = l2_policy(false);
#pragma unroll 1
    for (soff = 0; soff < p.nsteps && !dead; ++soff)
#pragma unroll 1
    for (int l = 0; l <= p.L && !dead; ++l) {
      const bool lm = l == p.L;
#pragma unroll 1
      for (int ph = 0; ph < 6 && !dead; ++ph) {
        int kind = -1;
        if (lm) {
          if (ph == 0 && p.V > 0) kind = K_LM;
        } else {
          switch (ph) {
            case 0: kind = K_QKV; break;
            case 1: issue_attn(l); kind = K_O; break;
            case 2: U = 0; kind = p.dense ? K_SHGU : K_ROUTER; break;
            case 3: kind = (!p.dense && p.nsh) ? K_SHGU : -1; break;
            case 4:
              if (!p.dense) {
                if (!routing(l, U, elist)) break;
                kind = K_RTGU;
              }
              break;
            default: kind = K_D; break;
          }
        }
        if (kind >= 0) issue_gemv(kind, lm ? 0 : l, U, elist);
      }
      if (!lm) ++lay;
    }
    // every copy this thread issued lands before it exits: consumers that gave up (an abort
    // elsewhere) no longer wait for their slots, and the CTA's shared memory must outlive them
    drain();
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
  unsigned item = 0;  // slots consumed so far in this step
  int rslot = 0;      // ring slot of the next item (item % ring, kept without divisions)
  unsigned rpar = 0;  // its full-barrier phase parity ((item / ring) & 1)
  bool dead = false;
  int warp, lane, tid;
  int stamp = 0;
  // Tile arithmetic: the tensor cores for steps of two or more tokens; at one token the CUDA
  // cores (a tensor-core MMA of M = 128 costs a fixed ~50 ns per K = 32 slice for any N <= 128,
  // so a 128 x 128 tile takes ~200 ns there, more than the ~160 ns of the CUDA-core product).
  static constexpr bool kTC = BM >= 2;
  bool range_bad = false;  // (CUDA-core path) an activation staged as f16 was outside its range
  // tensor-core tiles: tiles whose products were added so far in this step (the sequence picks
  // the TMEM accumulator and its barriers' phases), the TMEM base, the B operand layout
  unsigned ep = 0;    // this step's epoch (resident steps: the launch's epoch + steps done)
  int soff = 0;       // resident steps done in this launch
  unsigned gseq = 0;  // groups of tiles handed over so far (slot of TMEM slices, barrier phases)
  unsigned nstaged = 0;  // GEMV stages staged so far (thread 0)
  uint32_t tmem = 0;
  BGeo bg;

  __device__ Consumer(const KParams& p_, uint8_t* r, uint64_t* f, uint64_t* e, uint16_t* x, float* rd,
                      Misc* m_)
      : p(p_), ring(r), full(f), empty(e), xs(x), red(rd), m(m_) {
    tid = threadIdx.x;
    warp = tid >> 5;
    lane = tid & 31;
    bg = bgeo(p.B);
  }

  // CTA 0 records (event code, %globaltimer) pairs: code = what << 4 | event, where `what` is a
  // GEMV kind (0..6), 7 attention, 8 grid barrier, 9 routing wait, 10 step start/end, and event
  // 0 = begin, 1 = last tile consumed, 2 = finalisers done (barrier: its site number).
  __device__ void trace(int code) {
    if (DEC_TRACE && blockIdx.x == 0 && tid == 0 && stamp + 1 < kTraceSlots - kProducerTrace) {
      p.trace[stamp] = (unsigned long long)code;
      p.trace[stamp + 1] = gtimer();
      stamp += 2;
    }
  }

  // every CTA's time at dependency point k (a Stamp) of layer l < kStampLayers; only in a
  // library built with DEC_STAMPS=1 (the stores cost a few KB of code in every phase)
  __device__ void cta_stamp(int l, int k) {
    if (DEC_STAMPS && tid == 0 && l < kStampLayers)
      p.trace[kTraceSlots + ((size_t)l * kStampsPerLayer + k) * gridDim.x + blockIdx.x] = gtimer();
  }

  // Every consumer warp walks the same item sequence and takes part in every item (a GEMV tile
  // or a KV tile): a slot's "empty" barrier expects one arrival per consumer warp.
  __device__ const uint8_t* wait_item() {
    if (!dead) {
      if (!mbar_wait(&full[rslot], rpar, p, 20)) dead = true;
    }
    return ring + (size_t)rslot * kSlotBytes;
  }
  // release the current item's slot and move to the next item
  __device__ void release_item() {
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[rslot]);
    ++item;
    if (++rslot == p.ring) {
      rslot = 0;
      rpar ^= 1;
    }
  }

  // -------- activation staging --------

  __device__ const uint16_t* x_in(int l, int b) const {
    if (l > 0) return p.xbuf + ((size_t)(l & 1) * p.MB + b) * p.d;
    if (p.tokens) return p.embed + (size_t)m->tok[b] * p.d;
    return p.hidden_in + (size_t)b * p.d;
  }

  // xs[b][0..d) = bf16(rmsnorm(src_b) * w). The activation is read once (all loads of all
  // tokens issued together), parked in xs while the sums of squares are reduced, then scaled in
  // place.
  // With `from_o`, the input is x_mid = bf16(x_in + output projection), summed here from the
  // projection's published split-K partials (after every contributor has arrived).
  __device__ void stage_rmsnorm(int l_src, const uint16_t* direct, const uint16_t* w, bool from_o = false) {
    constexpr int MAXV = kMaxHidden / (kConsumerWarps * 32 * 8);  // 8-element chunks per thread
    const StageGeo go = stage_geo(p, K_O, 0);
    if (!direct && !from_o && l_src > 0) {
      // the previous layer's output rows (published by the down projection's finalisers)
      const unsigned* f = p.x_flag + (size_t)(l_src - 1) * p.n_rb_d;
      cta_wait_all(p.n_rb_d, [&](int rb) { return WaitCond{f + rb, ep}; }, 22);
      if (blockIdx.x == 0 && tid == 0) p.layer_ts[l_src] = gtimer();
    }
    if (from_o) {
      const int* cnt = p.cnt_o + (size_t)l_src * p.n_rb_d;
      cta_wait_all(p.n_rb_d, [&](int rb) {
        return count_reached(cnt + rb, (int)ep * go.kbs);
      }, 18);
      // Every output-projection tile has arrived, and each waited for the attention merges it
      // reads (together: all of layer l_src's), each merge having waited for all of its chunks.
      // So no CTA reads or adds to the layer's attention counters again in this launch: they
      // are zeroed here for the next one.
      if (tid == 0 && !dead) {
        for (int i = blockIdx.x; i < p.B * p.hkv; i += gridDim.x) p.attn_cnt[(size_t)l_src * p.MB * p.hkv + i] = 0;
        for (int g = blockIdx.x; g < p.hkv; g += gridDim.x) p.o_cnt[(size_t)l_src * p.hkv + g] = 0;
      }
    }
    // the norm weights of this thread's chunks, loaded once, in flight with the first activations
    uint4 wv[MAXV];
#pragma unroll
    for (int j = 0; j < MAXV; ++j) {
      const int k = (tid + j * kConsumerWarps * 32) * 8;
      if (k < p.d) wv[j] = __ldg(reinterpret_cast<const uint4*>(w + k));
    }
#pragma unroll 1
    for (int b = 0; b < min(p.B, BM); ++b) {
      const uint16_t* src = direct ? direct + (size_t)b * p.d : x_in(l_src, b);
      uint4 v[MAXV];
#pragma unroll
      for (int j = 0; j < MAXV; ++j) {
        const int k = (tid + j * kConsumerWarps * 32) * 8;
        if (k < p.d) v[j] = ldcg4(src + k);
      }
      if (from_o) {
        // the output projection's partials of this thread's chunks: two chunks at a time, six
        // contributors per batch, every load of a batch in flight before any is added (one L2
        // round trip per batch); each row is summed in contributor order
        const size_t st = (size_t)p.MB * kTileRows;
#pragma unroll
        for (int jp = 0; jp < MAXV; jp += 2) {  // MAXV == 2: one pass
          if ((tid + jp * kConsumerWarps * 32) * 8 >= p.d) break;
          float o8[2][8];
          int nc[2];
          const float* base[2];
#pragma unroll
          for (int jj = 0; jj < 2; ++jj) {
            const int k = (tid + (jp + jj) * kConsumerWarps * 32) * 8;
            const int rb = k / kTileRows;
            nc[jj] = k < p.d ? n_contrib(rb * go.kbs, go.kbs, go.T, gridDim.x) : 0;
            base[jj] = p.part_o + (size_t)rb * go.kbs * st + (size_t)b * kTileRows + k % kTileRows;
#pragma unroll
            for (int e = 0; e < 8; ++e) o8[jj][e] = 0.f;
          }
          const int ncm = max(nc[0], nc[1]);
          for (int c0 = 0; c0 < ncm; c0 += 6) {
            float4 t[2][6][2];
#pragma unroll
            for (int jj = 0; jj < 2; ++jj)
#pragma unroll
              for (int c = 0; c < 6; ++c) {
                if (c0 + c < nc[jj]) {
                  t[jj][c][0] = __ldcg(reinterpret_cast<const float4*>(base[jj] + (size_t)(c0 + c) * st));
                  t[jj][c][1] = __ldcg(reinterpret_cast<const float4*>(base[jj] + (size_t)(c0 + c) * st + 4));
                } else {
                  t[jj][c][0] = t[jj][c][1] = make_float4(0.f, 0.f, 0.f, 0.f);
                }
              }
#pragma unroll
            for (int jj = 0; jj < 2; ++jj)
#pragma unroll
              for (int c = 0; c < 6; ++c) {
                o8[jj][0] += t[jj][c][0].x; o8[jj][1] += t[jj][c][0].y; o8[jj][2] += t[jj][c][0].z; o8[jj][3] += t[jj][c][0].w;
                o8[jj][4] += t[jj][c][1].x; o8[jj][5] += t[jj][c][1].y; o8[jj][6] += t[jj][c][1].z; o8[jj][7] += t[jj][c][1].w;
              }
          }
#pragma unroll
          for (int jj = 0; jj < 2; ++jj) {
            if ((tid + (jp + jj) * kConsumerWarps * 32) * 8 < p.d) {
              uint32_t* u = reinterpret_cast<uint32_t*>(&v[jp + jj]);
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                const uint16_t lo = f2bf(bf16lo(u[q]) + o8[jj][2 * q]);
                const uint16_t hi = f2bf(bf16hi(u[q]) + o8[jj][2 * q + 1]);
                u[q] = (uint32_t)lo | ((uint32_t)hi << 16);
              }
            }
          }
        }
      }
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
          if constexpr (kTC) park(b, k, v[j]);
          else *reinterpret_cast<uint4*>(xs + (size_t)b * p.xmax + k) = v[j];
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      if (lane == 0) m->rsum[warp][b] = ss;
    }
    cons_sync();
#pragma unroll 1
    for (int b = 0; b < min(p.B, BM); ++b) {
      float ss = 0.f;
#pragma unroll
      for (int wi = 0; wi < kConsumerWarps; ++wi) ss += m->rsum[wi][b];
      const float inv = 1.0f / sqrtf(ss / (float)p.d + p.eps);
#pragma unroll
      for (int j = 0; j < MAXV; ++j) {
        const int k = (tid + j * kConsumerWarps * 32) * 8;
        const bool in = k < p.d;  // (whole half-warps: d is a multiple of 128)
        float f[8];
        if (in) {
          const uint4 xv = kTC ? unpark(b, k) : *reinterpret_cast<const uint4*>(xs + (size_t)b * p.xmax + k);
          const uint32_t* u = reinterpret_cast<const uint32_t*>(&xv);
          const uint32_t* wu = reinterpret_cast<const uint32_t*>(&wv[j]);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            f[2 * q] = bf16f(f2bf((bf16lo(u[q]) * inv) * bf16lo(wu[q])));
            f[2 * q + 1] = bf16f(f2bf((bf16hi(u[q]) * inv) * bf16hi(wu[q])));
          }
        }
        if constexpr (kTC) {
          pieces(b, k, f, in);
        } else if (in) {
          *reinterpret_cast<uint4*>(xs + (size_t)b * p.xmax + k) =
              make_uint4(pack_f16x2(f[0], f[1]), pack_f16x2(f[2], f[3]), pack_f16x2(f[4], f[5]), pack_f16x2(f[6], f[7]));
        }
      }
    }
    if constexpr (kTC) fence_proxy_async_smem();
    else range_check();
    cons_sync();
  }

  // (CUDA-core path) The GEMV input is staged in shared memory as f16: every bf16 value with
  // magnitude in [2^-17, 65504] converts exactly (8 significant bits fit in f16's 11); smaller
  // ones round with an absolute error below 2^-25, far under the fp32 accumulation error of the
  // sums they feed. A value beyond the f16 range would become infinite, so it is reported as a
  // device error. (The range test only sets a per-thread flag; range_check() reports it once per
  // staging.)
  __device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    range_bad |= !(fabsf(lo) <= 65504.f) || !(fabsf(hi) <= 65504.f);
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
  }
  __device__ __forceinline__ void range_check() {
    if (range_bad) {
      raise_err(p, kDevRange, 5);
      range_bad = false;
    }
  }

  // ---- the tensor cores' B operand (the stage's activations as E4M3 pieces)

  // byte of activation k (of the stage's input) of token b, piece r, in the B operand layout
  __device__ __forceinline__ uint8_t* bpos(int b, int k, int r) const {
    const int kb = k >> 7, c = k & 127;
    const int row = (kb % bg.pk) * bg.rpad + 2 * b + r;
    return reinterpret_cast<uint8_t*>(xs) + (size_t)(kb / bg.pk) * bg.nrb * 128 + (row >> 3) * 1024 + (c >> 4) * 128 +
           (row & 7) * 16 + (c & 15);
  }
  // Park 8 bf16 activations k .. k + 7 of token b where their pieces will go: low bytes at piece
  // 0's place, high bytes at piece 1's (so converting them later in place touches no other
  // thread's data); unpark reads them back.
  __device__ __forceinline__ void park(int b, int k, const uint4 v) {
    *reinterpret_cast<uint2*>(bpos(b, k, 0)) = make_uint2(__byte_perm(v.x, v.y, 0x6420), __byte_perm(v.z, v.w, 0x6420));
    *reinterpret_cast<uint2*>(bpos(b, k, 1)) = make_uint2(__byte_perm(v.x, v.y, 0x7531), __byte_perm(v.z, v.w, 0x7531));
  }
  __device__ __forceinline__ uint4 unpark(int b, int k) const {
    const uint2 lo = *reinterpret_cast<const uint2*>(bpos(b, k, 0));
    const uint2 hi = *reinterpret_cast<const uint2*>(bpos(b, k, 1));
    return make_uint4(__byte_perm(lo.x, hi.x, 0x5140), __byte_perm(lo.x, hi.x, 0x7362), __byte_perm(lo.y, hi.y, 0x5140),
                      __byte_perm(lo.y, hi.y, 0x7362));
  }
  // Activations k .. k + 7 of token b (bf16 values in f) as two E4M3 pieces each: with 2^a
  // putting the largest |x| of their k block (the 16 chunks of a half-warp) in [128, 256),
  // x * 2^a = p1 + p2 / 16, p1 = E4M3(x * 2^a), p2 = E4M3(16 (x * 2^a - p1)); exact for
  // |x| >= 2^-13 max|x| (the residual has at most 4 significant bits), an error below
  // 2^-21 max|x| under it. Called by whole warps (the maximum is a half-warp shuffle).
  __device__ __forceinline__ void pieces(int b, int k, const float (&f)[8], bool in) {
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
    *reinterpret_cast<uint2*>(bpos(b, k, 0)) = make_uint2(w1[0], w1[1]);
    *reinterpret_cast<uint2*>(bpos(b, k, 1)) = make_uint2(w2[0], w2[1]);
    if ((lane & 15) == 0) m->xexp[b][k >> 7] = (int8_t)a;
  }

  // Stage activations dst_off .. dst_off + n of the stage's input (as B operand pieces) from a
  // bf16 activation src[b][0..n) written by other CTAs; two 8-element chunks per thread and
  // pass, both loads in flight before either is converted. n and dst_off are multiples of 128.
  __device__ void stage_copy(const uint16_t* src, int n, size_t src_stride, int dst_off) {
    constexpr int P = kConsumerWarps * 32 * 8;
#pragma unroll 1
    for (int b = 0; b < min(p.B, BM); ++b) {
#pragma unroll 1
      for (int k0 = (tid & ~31) * 8; k0 < n; k0 += 2 * P) {  // (whole warps take part)
        const int k = k0 + lane * 8;
        uint4 v[2];
#pragma unroll
        for (int j = 0; j < 2; ++j)
          if (k + j * P < n) v[j] = ldcg4(src + (size_t)b * src_stride + k + j * P);
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const bool in = k + j * P < n;
          float f[8];
          if (in) {
            const uint32_t* u = reinterpret_cast<const uint32_t*>(&v[j]);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              f[2 * q] = bf16lo(u[q]);
              f[2 * q + 1] = bf16hi(u[q]);
            }
          }
          if constexpr (kTC) {
            pieces(b, dst_off + k + j * P, f, in);
          } else if (in) {
            *reinterpret_cast<uint4*>(xs + (size_t)b * p.xmax + dst_off + k + j * P) =
                make_uint4(pack_f16x2(f[0], f[1]), pack_f16x2(f[2], f[3]), pack_f16x2(f[4], f[5]),
                           pack_f16x2(f[6], f[7]));
          }
        }
      }
    }
    if constexpr (kTC) fence_proxy_async_smem();
    else range_check();
  }

  // -------- split-K GEMV over one stage, on the tensor cores --------

  // A tile (128 weight rows x 128 E4M3 columns, repacked in the canonical K-major layout: 8-row x
  // 16-byte core matrices, 128 bytes apart along K and 1024 apart along the rows) is multiplied
  // straight from its ring slot by tcgen05.mma kind::f8f6f4 (issued by the MMA warp): A = the raw
  // E4M3 codes, B = the stage's bf16 activations split exactly into two E4M3 pieces per value
  // (see pieces()), D = 128 rows x 16 fp32 columns in the tile's own TMEM slice. Products of
  // 8-bit values are exact and the sums are fp32. The consumer warps add each tile's product
  // into fp32 registers, applying the pieces' scales, the tile's block scale and the expert gate
  // (a k block per tile, so the block scale cannot stay in TMEM). The tensor cores replace the
  // E4M3 conversions that bound a CUDA-core dot product.

  // (CUDA-core path, one token) All eight consumer warps share each tile: warp w takes row
  // R = 32 (w & 3) + lane and the 16-byte column chunks 4 (w >> 2) .. + 3 (chunk c of row R sits
  // at 16 ((R / 8 * 8 + c) * 8 + R % 8) in the tensor cores' layout: each load of a warp reads
  // four 128-byte runs, no bank conflict beyond the 512 bytes' minimum). E4M3 pairs become f16
  // pairs exactly (CUDA's cvt); each product is formed and accumulated in fp32 by one mixed-
  // precision FMA (f16 x f16 + f32, one rounding). The block scale of the row's half multiplies
  // the tile sum. The activation chunk is the same for all lanes (a broadcast load).
  __device__ __forceinline__ void tile_dot(const uint8_t* tile, int xoff, const float* gmul, float (&acc)[4]) {
    const int r = warp & 3, c0 = (warp >> 2) * 4, R = 32 * r + lane;
    const float2 sc = *reinterpret_cast<const float2*>(tile + kTileData);
    const float s_r = r < 2 ? sc.x : sc.y;
    float part[BM][2];  // two FMA chains per token
#pragma unroll
    for (int b = 0; b < BM; ++b) part[b][0] = part[b][1] = 0.f;
    uint4 wv[4];
#pragma unroll
    for (int c = 0; c < 4; ++c)
      wv[c] = *reinterpret_cast<const uint4*>(tile + ((((R >> 3) * 8 + c0 + c) * 8 + (R & 7)) << 4));
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const uint32_t* u = reinterpret_cast<const uint32_t*>(&wv[c]);
      uint32_t wh[8];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        wh[2 * j] = e4m3x2_to_f16x2(u[j]);
        wh[2 * j + 1] = e4m3x2_to_f16x2(u[j] >> 16);
      }
#pragma unroll
      for (int b = 0; b < BM; ++b) {
        if (b < p.B) {
          const uint16_t* xp = xs + (size_t)b * p.xmax + xoff + (c0 + c) * 16;
          const uint4 x0 = *reinterpret_cast<const uint4*>(xp);
          const uint4 x1 = *reinterpret_cast<const uint4*>(xp + 8);
          const uint32_t xh[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
          for (int j = 0; j < 8; ++j) fma_f16x2_f32(wh[j], xh[j], part[b][0], part[b][1]);
        }
      }
    }
#pragma unroll
    for (int b = 0; b < BM && b < 4; ++b) acc[b] = fmaf(s_r * gmul[b], part[b][0] + part[b][1], acc[b]);
  }

  // Add the products of group gs (n consecutive tiles of one segment, from position pos) into the
  // thread's accumulators. Thread (warp w, lane) holds row 32 (w & 3) + lane of tokens
  // 4 (w >> 2) .. 4 (w >> 2) + 3 (TMEM lane quadrant w & 3; tile i's product is slice
  // (group slot) * kGT + i, where token b's pieces are columns cb + 2b, cb + 2b + 1 for its k
  // block kbi, cb = (kbi mod pk) rpad), scaled by the pieces' 2^-a, the tile's block scale (copied
  // by the MMA warp) and the expert gate. Every consumer warp then hands the slices back.
  __device__ void group_epilogue(unsigned gs, int n, TilePos pos, int kind, int nv, const StageGeo& g,
                                 float (&acc)[4]) {
    const int gsl = gs % kNG;
    if (!dead && !mbar_wait(&m->tfull[gsl], (gs / kNG) & 1, p, 25)) dead = true;
    const int q = warp & 3, h = warp >> 2;
    if (!dead && 4 * h < p.B) {  // (warp-uniform)
      tc_fence_after();
      const int row = 32 * q + lane;
      constexpr int NC = BM >= 4 ? 8 : 2 * BM;
#pragma unroll 1
      for (int i = 0; i < n; ++i) {
        const int kbi = pos.kbi(p, kind);
        const float2 sc = m->hdr[gsl][i];
        const float s_r = row < 64 ? sc.x : sc.y;
        const uint32_t ta = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)((gsl * kGT + i) * kMmaN) +
                            (uint32_t)((kbi % bg.pk) * bg.rpad + 8 * h);
        float d[8];
        tmem_ld<NC>(ta, d);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int b = 4 * h + j;
          if (b < p.B && 2 * j < NC) {
            const float gm = kind == K_D ? m->gate[b][min(pos.v, kMaxExperts)] : 1.f;
            const float inv = __int_as_float((127 - (int)m->xexp[b][kbi]) << 23);  // 2^-a
            acc[j] = fmaf(s_r * gm * inv, fmaf(d[2 * j + 1], 0.0625f, d[2 * j]), acc[j]);
          }
        }
        pos.next(p, g, kind, nv);
      }
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&m->tempty[gsl]);
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

  // Cross-warp reduction of one segment's accumulators, publication of the CTA's partial sums,
  // and the arrival on the output group's counter (result kept for the end of the stage).
  __device__ int* pub_counter(int kind, int l) const {
    if (kind == K_ROUTER) return p.cnt_router + l;
    return kind == K_QKV ? p.cnt_qkv + (size_t)l * p.n_rb_qkv : p.cnt_o + (size_t)l * p.n_rb_d;
  }

  // output groups of a finalised stage (SwiGLU row blocks of each expert, output row blocks,
  // vocabulary row blocks)
  __device__ __forceinline__ int n_groups(int kind, const StageGeo& g) const {
    return kind == K_D ? p.n_rb_d : g.T / g.kbs;  // down projections: the output row blocks
  }

  __device__ void flush(int kind, int l, const StageGeo& g, int seg, int first_tile, int ntiles, float (&acc)[4]) {
    const int row_t = 32 * (warp & 3) + lane, h = warp >> 2;
    if constexpr (kTC) {
      // red[row][b]: thread (warp w, lane) holds row 32 (w & 3) + lane of tokens 4 (w >> 2) + i
#pragma unroll
      for (int i = 0; i < 4; ++i)
        if (4 * h + i < BM) red[(size_t)row_t * BM + 4 * h + i] = acc[i];
    } else {
      // red[column half][row][b]: the two column halves of a row are summed below
#pragma unroll
      for (int b = 0; b < BM && b < 4; ++b) red[((size_t)h * kTileRows + row_t) * BM + b] = acc[b];
    }
    cons_sync();
    const int a = seg * g.kbs;
    const int slot = contrib_slot(blockIdx.x, first_tile, a, g.T, gridDim.x);
    float* dst = part_base(kind) + ((size_t)seg * g.kbs + slot) * p.MB * kTileRows;
    #pragma unroll 1
    for (int idx = tid; idx < p.B * kTileRows; idx += kConsumerWarps * 32) {
      const int b = idx / kTileRows, row = idx % kTileRows;
      dst[(size_t)b * kTileRows + row] = kTC ? red[(size_t)row * BM + b]
                                             : red[(size_t)row * BM + b] + red[((size_t)kTileRows + row) * BM + b];
    }
    // The CTA barrier orders every thread's partial before the publishing thread's releasing
    // arrival; no other thread waits for the arrival to complete. An arrival adds the number of
    // the segment's tiles the CTA summed, so a group is complete when its counter has grown by
    // its tile count (kbs per segment), however the tiles were split among the CTAs.
    cons_sync();
    if (dead) return;
    if (kind == K_QKV || kind == K_O || kind == K_ROUTER) {
      // published partials: the readers wait for all of the row block's tiles (in tests, the
      // CTA holding the first q/k/v tile may withhold that arrival in layer 0, so waits run out)
      const bool withhold = p.test_skip && kind == K_QKV && l == 0 && first_tile == 0;
      if (tid == kPubThread && !withhold) red_release_add(pub_counter(kind, l) + seg, ntiles);
      return;
    }
    // (expert-major down projections: segment v * n_rb_d + rb adds to output row block rb)
    if (tid == kPubThread) red_release_add(cnt_base(kind) + (kind == K_D && !g.rbm ? seg % p.n_rb_d : seg), ntiles);
  }

  // counter value that completes an output group: its segment's tiles
  // (down projections: every expert slot's k blocks of the row block, in either tile order)
  __device__ int group_expected(int kind, const StageGeo& g, int grp) const {
    return kind == K_D ? g.T / p.n_rb_d : g.kbs;
  }

  // sum of the published partials of segment seg for (b, row)
  __device__ __forceinline__ float seg_sum(int kind, const StageGeo& g, int seg, int b, int row) const {
    const int nc = n_contrib(seg * g.kbs, g.kbs, g.T, gridDim.x);
    const float* src = part_base(kind) + (size_t)seg * g.kbs * p.MB * kTileRows + (size_t)b * kTileRows + row;
    const size_t st = (size_t)p.MB * kTileRows;
    float s = 0.f;
#pragma unroll 1
    for (int c0 = 0; c0 < nc; c0 += 8) {  // eight independent loads in flight, summed in slot order
      float v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = (c0 + j < nc) ? ldcg(src + (size_t)(c0 + j) * st) : 0.f;
#pragma unroll
      for (int j = 0; j < 8; ++j) s += v[j];
    }
    return s;
  }

  // seg_sum of two rows of one segment, with both rows' loads of a batch in flight together
  __device__ __forceinline__ void seg_sum2(int kind, const StageGeo& g, int seg, int b, int r0, int r1, float& s0,
                                           float& s1) const {
    const int nc = n_contrib(seg * g.kbs, g.kbs, g.T, gridDim.x);
    const float* src = part_base(kind) + (size_t)seg * g.kbs * p.MB * kTileRows + (size_t)b * kTileRows;
    const size_t st = (size_t)p.MB * kTileRows;
    s0 = s1 = 0.f;
    for (int c0 = 0; c0 < nc; c0 += 8) {
      float v0[8], v1[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        v0[j] = (c0 + j < nc) ? ldcg(src + (size_t)(c0 + j) * st + r0) : 0.f;
        v1[j] = (c0 + j < nc) ? ldcg(src + (size_t)(c0 + j) * st + r1) : 0.f;
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        s0 += v0[j];
        s1 += v1[j];
      }
    }
  }

  __device__ void gemv_stage(int kind, int l, int U) {
    const StageGeo g = stage_geo(p, kind, U);
    const int G_ = gridDim.x;
    const int t0 = range_lo(g.T, blockIdx.x, G_), t1 = range_lo(g.T, blockIdx.x + 1, G_);
    cons_sync();  // the stage's activations are staged (and fenced for the tensor cores)
    if (kTC && tid == 0) {
      ++nstaged;
      __threadfence_block();
      *reinterpret_cast<volatile unsigned*>(&m->stages_staged) = nstaged;
    }
    trace(kind << 4);
    float gmul[BM];
    float acc[4];
    int seg_cur = -1, seg_first = 0;
    // Position of tile t, advanced without divisions: segment, k block within it, and for the
    // down projection the expert slot v (whose gates scale the tile), the k block kx within its
    // run and the expert's place xj among the SwiGLU rows staged (the CTA's runs in order, the
    // first at 0, wrapping after nv). The MMA warp walks the same positions.
    const int nv = kind == K_D ? U + p.nsh : 1;
    TilePos pe;
    pe.init(p, g, kind, t0, t1);
    int j = 0;  // tile j of the current slot (the producer packs kSlotTiles consecutive tiles per slot)
    const uint8_t* slot_base = ring;
    for (int t = t0;;) {
      // a segment ends at a segment boundary or at the end of the range (one flush call site)
      if (t == t1 || pe.seg != seg_cur) {
        if (t == t1) {
          // one verdict for the whole CTA: a thread may have given up on a wait that another
          // thread saw end, and the finalisers below branch on it around barriers
          dead = cons_any(dead);
          trace(kind << 4 | 1);
          if (kind == K_QKV) cta_stamp(l, S_QKV_TILES);
          if (kind == K_O) cta_stamp(l, S_O_TILES);
          if (kind == K_RTGU || (kind == K_SHGU && p.dense)) cta_stamp(l, S_GU_TILES);
          if (kind == K_D) cta_stamp(l, S_D_TILES);
        }
        if (seg_cur >= 0) flush(kind, l, g, seg_cur, seg_first, t - seg_first, acc);
        if (t == t1) break;
        seg_cur = pe.seg;
        seg_first = t;
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[i] = 0.f;
      }
      if constexpr (kTC) {
        // a group: up to kGT tiles of this segment (the MMA warp forms the same groups)
        const int n = min(kGT, min(t1, (pe.seg + 1) * g.kbs) - t);
        group_epilogue(gseq++, n, pe, kind, nv, g, acc);
        for (int i = 0; i < n; ++i) pe.next(p, g, kind, nv);
        t += n;
      } else {
#pragma unroll
        for (int b = 0; b < BM; ++b) gmul[b] = kind == K_D ? m->gate[b][min(pe.v, kMaxExperts)] : 1.f;
        if (j == 0) slot_base = wait_item();
        if (!dead) tile_dot(slot_base + (size_t)j * kTileBytes, pe.kbi(p, kind) * kTileK, gmul, acc);
        if (++j == kSlotTiles || t == t1 - 1) {
          release_item();
          j = 0;
        }
        pe.next(p, g, kind, nv);
        ++t;
      }
    }
    if constexpr (kTC) {
      // the stage's weight slots were freed by the MMA warp; keep the ring position in step
      for (int k = 0; k < (t1 - t0 + kSlotTiles - 1) / kSlotTiles; ++k) {
        ++item;
        if (++rslot == p.ring) {
          rslot = 0;
          rpar ^= 1;
        }
      }
    }
    // Finalise the output groups this CTA is designated for (groups spread evenly over the
    // CTAs, so no CTA finalises two while others finalise none): wait (acquire) until every
    // contributor has arrived, reset the counter for the next launch or layer (before the
    // result is published, and nothing else touches it before then: every later arrival on it
    // depends on this group's result), finalise. No contributor ever waits for the result of its
    // own arrival.
    // The SwiGLU groups of an MoE layer, routed experts' and shared experts' alike, are all
    // finalised after the routed gate/up stage, together (see finalize_gu): a CTA designated for
    // a shared-expert group then does not start its routed tiles late.
    const bool gu = kind == K_RTGU || (kind == K_SHGU && p.dense);
    int ng = 0;
    if (kind == K_RTGU) ng = (U + (p.nsh ? 1 : 0)) * p.n_rb_gu;
    else if (gu || kind == K_D || kind == K_LM) ng = n_groups(kind, g);
    const int f_lo = (int)(((long long)blockIdx.x * ng + G_ - 1) / G_);
    const int f_hi = (int)(((long long)(blockIdx.x + 1) * ng + G_ - 1) / G_);
    if (gu) {
      if (f_hi > f_lo && !dead) finalize_gu(l, f_lo, f_hi, U);
    } else {
      for (int grp = f_lo; grp < f_hi && !dead; ++grp) {
        const int* c = cnt_base(kind) + grp;
        const int want = group_expected(kind, g, grp);
        cta_wait_all(1, [&](int) { return count_reached(c, want); }, 21);
        if (dead) break;
        if (tid == kPubThread) *const_cast<volatile int*>(c) = 0;
        finalize(kind, l, g, grp, U);
        cons_sync();
      }
    }
    trace(kind << 4 | 2);
  }

  // -------- routing (every CTA computes it) --------

  // Routing of layer l from the router's published partials: logits -> per-token top-k (ties to
  // the lower expert index) -> sigmoid scores normalised over the selection -> the distinct
  // experts in ascending order (m->elist, m->U) and each token's gate per distinct expert
  // (m->gate). Every CTA computes the same result (same partials, same order), so no CTA waits
  // for another one's selection; the CTA's producer is told through the routing mbarrier.
  // CTA 0 also writes the selections for inspection.
  __device__ void local_routing(int l) {
    const StageGeo g = stage_geo(p, K_ROUTER, 0);
    const int nc = n_contrib(0, g.kbs, g.T, gridDim.x);
    const int* cnt = p.cnt_router + l;
    cta_wait_all(1, [&](int) { return count_reached(cnt, (int)ep * g.kbs); }, 19);
    float* tmp = red;                                        // [BM][128] logits
    int* mark = reinterpret_cast<int*>(tmp + BM * kTileRows);  // [128] rank + 1 of expert e
    int* sel = mark + kMaxExperts;                              // [BM][16]
    float* sg = reinterpret_cast<float*>(sel + BM * 16);        // [BM][16]
    // logits: TPI threads per (token, expert) sum interleaved contributor subsets, eight loads
    // in flight per batch, then combine with a fixed butterfly (deterministic order)
    {
      const int items = p.B * p.E;
      int tpi = 1;
      while (tpi < 8 && tpi * 2 * items <= kConsumerWarps * 32) tpi *= 2;
      const size_t st = (size_t)p.MB * kTileRows;
      const int per = kConsumerWarps * 32 / tpi;  // items handled per pass
      for (int i0 = 0; i0 < items; i0 += per) {
        const int it = i0 + tid / tpi, part = tid % tpi;
        const int b = it / max(p.E, 1), e = it % max(p.E, 1);
        const bool ok = it < items;
        const float* src = p.part_router + (size_t)b * kTileRows + e;
        float s = 0.f;
        for (int c0 = part; c0 < nc; c0 += 8 * tpi) {
          float v[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) v[j] = (ok && c0 + j * tpi < nc) ? ldcg(src + (size_t)(c0 + j * tpi) * st) : 0.f;
#pragma unroll
          for (int j = 0; j < 8; ++j) s += v[j];
        }
        for (int o = 1; o < tpi; o <<= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if (ok && part == 0) tmp[b * kTileRows + e] = s;
      }
      for (int idx = tid; idx < BM * kTileRows; idx += kConsumerWarps * 32) {
        const int b = idx / kTileRows, e = idx % kTileRows;
        if (b >= p.B || e >= p.E) tmp[idx] = -INFINITY;
      }
    }
    if (tid < kMaxExperts) mark[tid] = 0;
    cons_sync();
    // top-k by rank: thread (b, e) counts the experts ahead of e (a larger logit, or an equal
    // one at a lower index; a NaN logit counts as -inf, so the order is total and the ranks of a
    // token are a permutation). Ranks 0..top_k-1 are the selection, in descending order.
#pragma unroll 1
    for (int idx = tid; idx < p.B * p.E; idx += kConsumerWarps * 32) {
      const int b = idx / p.E, e = idx - b * p.E;
      const float* row = tmp + b * kTileRows;
      float v = row[e];
      if (blockIdx.x == 0) p.rt_logits[((size_t)l * p.rows + b) * p.E + e] = v;  // for inspection
      if (v != v) v = -INFINITY;
      int rank = 0;
#pragma unroll 4
      for (int j = 0; j < p.E; ++j) {
        float w = row[j];
        if (w != w) w = -INFINITY;
        rank += (w > v || (w == v && j < e)) ? 1 : 0;
      }
      if (rank < p.topk) {
        sel[b * 16 + rank] = e;
        sg[b * 16 + rank] = 1.0f / (1.0f + expf(-v));
        mark[e] = 1;
      }
    }
    cons_sync();
    if (warp < p.B) {
      // gates: the selected scores over their sum (taken in rank order)
      const int b = warp;
      float ssum = 0.f;
#pragma unroll 1
      for (int k = 0; k < p.topk; ++k) ssum += sg[b * 16 + k];
      __syncwarp();
      if (lane < p.topk) {
        const float gt = sg[b * 16 + lane] / ssum;
        sg[b * 16 + lane] = gt;
        if (blockIdx.x == 0) {
          p.rt_idx[((size_t)l * p.rows + b) * p.topk + lane] = sel[b * 16 + lane];
          p.rt_topk_gate[((size_t)l * p.rows + b) * p.topk + lane] = gt;
        }
      }
    }
    cons_sync();
    if (warp == 0) {
      // distinct experts in ascending order: ballot prefix over the marks
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
      if (lane == 0) m->U = min(U2, p.umax);
    }
    for (int idx = tid; idx < BM * (kMaxExperts + 1); idx += kConsumerWarps * 32)
      m->gate[idx / (kMaxExperts + 1)][idx % (kMaxExperts + 1)] = 0.f;
    cons_sync();
    for (int idx = tid; idx < p.B * p.topk; idx += kConsumerWarps * 32) {
      const int b = idx / p.topk, k = idx % p.topk;
      const int e = sel[b * 16 + k];
      m->gate[b][mark[e] - 1] = sg[b * 16 + k];
    }
    cons_sync();
    if (tid == 0) mbar_arrive(&m->rt_bar);  // the producer may now issue the routed experts
    // The SwiGLU counters h_cnt[l][slot] grow by n_rb_gu per step for every slot (so a wait's
    // target is epoch * n_rb_gu whatever the slot did in earlier steps): the slots this step's
    // routing leaves unused get their n_rb_gu here, spread over the CTAs.
    if (tid == kPubThread)
      for (int u = m->U + blockIdx.x; u < p.umax; u += gridDim.x)
        red_relaxed_add(p.h_cnt + (size_t)l * (p.umax + 1) + u, p.n_rb_gu);
  }

  // -------- finalisers (run by the CTA designated for an output group) --------

  // SwiGLU of the gate/up groups vlo..vhi-1 of layer l, all at once: one wait for all of their
  // counters, one pass over their rows. Groups v < U * n_rb_gu are routed (expert slot
  // v / n_rb_gu, row block v % n_rb_gu), the rest the shared experts' (or the dense FFN's) row
  // blocks. Each row block holds 64 gate rows then the matching 64 up rows;
  // h = bf16(silu(gate) * up) from the contributor partials summed in slot order.
  __device__ void finalize_gu(int l, int vlo, int vhi, int U) {
    const int half = kTileRows / 2;
    const int nr = U * p.n_rb_gu;
    const StageGeo gr = stage_geo(p, K_RTGU, U), gs = stage_geo(p, K_SHGU, 0);
    cta_wait_all(vhi - vlo, [&](int i) {
      const int v = vlo + i;
      return v < nr ? count_reached(p.cnt_rtgu + v, group_expected(K_RTGU, gr, v))
                    : count_reached(p.cnt_shgu + (v - nr), group_expected(K_SHGU, gs, v - nr));
    }, 21);
    if (dead) return;
    if (tid == kPubThread) {
#pragma unroll 1
      for (int v = vlo; v < vhi; ++v) *const_cast<volatile int*>(v < nr ? p.cnt_rtgu + v : p.cnt_shgu + (v - nr)) = 0;
    }
    const int per = p.B * half;
#pragma unroll 1
    for (int idx = tid; idx < (vhi - vlo) * per; idx += kConsumerWarps * 32) {
      const int v = vlo + idx / per, r = idx % per;
      const int b = r / half, i = r % half;
      const bool sh = v >= nr;
      const int grp = sh ? v - nr : v;
      float gv, uv;
      seg_sum2(sh ? K_SHGU : K_RTGU, sh ? gs : gr, grp, b, i, i + half, gv, uv);
      const uint16_t h = f2bf((gv / (1.0f + expf(-gv))) * uv);
      const int j = (sh ? grp : grp % p.n_rb_gu) * half + i;
      if (sh)
        p.hsh[(size_t)b * p.inter + j] = h;
      else
        p.hrt[((size_t)(grp / p.n_rb_gu) * p.MB + b) * p.inter + j] = h;
    }
    cons_sync();
    if (tid == kPubThread) {
      // one arrival per group on its expert slot's counter h_cnt[l][slot] (slot v / n_rb_gu, the
      // shared experts' umax), which grows by n_rb_gu per step
      int* c = p.h_cnt + (size_t)l * (p.umax + 1);
#pragma unroll 1
      for (int v = vlo; v < vhi; ++v) red_release_add(c + (v < nr ? v / p.n_rb_gu : p.umax), 1);
    }
  }

  // Output-projection row block (D: residual + down projections) or LM-head block grp.

  __device__ void finalize(int kind, int l, const StageGeo& g, int grp, int U) {
    float* tmp = red;  // [BM][128]
    switch (kind) {
      case K_D: {
        // the row block's contributor slots (partial rows of part_d): one run of consecutive
        // slots (row-block major), or one run per expert slot (expert major), listed by warp 0
        // (lane v counts run v's contributors, a prefix sum places them)
        int* list = reinterpret_cast<int*>(tmp + BM * kTileRows);
        int* nlist = list + kListCap;
        const int rb0 = grp * g.kbs;  // row-block major: the slots rb0 .. rb0 + nl - 1
        if (!g.rbm && warp == 0) {
          const int nseg = g.T / g.tpe;
          int base = 0;
#pragma unroll 1
          for (int v0 = 0; v0 < nseg; v0 += 32) {
            const int v = v0 + lane;
            const int seg = v * p.n_rb_d + grp;
            const int nc = v < nseg ? n_contrib(seg * g.kbs, g.kbs, g.T, gridDim.x) : 0;
            int incl = nc;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
              const int y = __shfl_up_sync(0xffffffffu, incl, o);
              if (lane >= o) incl += y;
            }
            const int first = base + incl - nc;
#pragma unroll 1
            for (int c = 0; c < nc; ++c)
              if (first + c < kListCap) list[first + c] = seg * g.kbs + c;
            base += __shfl_sync(0xffffffffu, incl, 31);
          }
          if (lane == 0) {
            if (base > kListCap) raise_err(p, kDevBadArg, 3);
            *nlist = min(base, kListCap);
          }
        }
        if (!g.rbm) cons_sync();
        const int nl = g.rbm ? n_contrib(rb0, g.kbs, g.T, gridDim.x) : *nlist;
        const StageGeo go = stage_geo(p, K_O, 0);
        const int nco = n_contrib(grp * go.kbs, go.kbs, go.T, gridDim.x);
        const size_t st = (size_t)p.MB * kTileRows;
#pragma unroll 1
        for (int idx = tid; idx < p.B * kTileRows; idx += 256) {
          int b = idx / kTileRows, i = idx % kTileRows;
          int r = grp * kTileRows + i;
          const float* src = p.part_d + (size_t)b * kTileRows + i;
          const float* osrc = p.part_o + (size_t)grp * go.kbs * st + (size_t)b * kTileRows + i;
          // the residual input, the output projection's partials (x_mid, as the norm stage
          // formed it) and the first eight down-projection partials, all in flight together
          const uint16_t xin = ldcg_u16(x_in(l, b) + r);
          float ov[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) ov[j] = (j < nco) ? ldcg(osrc + (size_t)j * st) : 0.f;
          float y = 0.f;
#pragma unroll 1
          for (int e0 = 0; e0 < nl; e0 += 8) {  // eight contributors per batch, in list order
            float v[8];
#pragma unroll
            for (int j = 0; j < 8; ++j)
              v[j] = (e0 + j < nl) ? ldcg(src + (size_t)(g.rbm ? rb0 + e0 + j : list[e0 + j]) * st) : 0.f;
#pragma unroll
            for (int j = 0; j < 8; ++j) y += v[j];
          }
          float os = 0.f;
#pragma unroll
          for (int j = 0; j < 8; ++j) os += ov[j];
#pragma unroll 1
          for (int c = 8; c < nco; ++c) os += ldcg(osrc + (size_t)c * st);
          const float xm = bf16f(f2bf(bf16f(xin) + os));
          uint16_t o = f2bf(xm + y);
          p.xbuf[((size_t)((l + 1) & 1) * p.MB + b) * p.d + r] = o;
          if (l == p.L - 1 && p.hidden_out) p.hidden_out[(size_t)b * p.d + r] = o;
        }
        // the next layer's input row block is final
        cons_sync();
        if (tid == kPubThread) st_release(p.x_flag + (size_t)l * p.n_rb_d + grp, ep);
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
        // warp b: the block's largest logit of token b, ties to the lower row (each lane scans
        // its rows in ascending order, the butterfly keeps the lower row of equal values)
#pragma unroll 1
        for (int b = warp; b < p.B; b += kConsumerWarps) {
          float bv = tmp[b * kTileRows + lane];
          int bi = lane;
#pragma unroll
          for (int j = 1; j < kTileRows / 32; ++j) {
            const float x = tmp[b * kTileRows + lane + 32 * j];
            if (x > bv) { bv = x; bi = lane + 32 * j; }
          }
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
            if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
          }
          if (lane == 0)
            atomicMax(p.amax + b, ((unsigned long long)float_key(bv) << 32) |
                                      (unsigned long long)(0xFFFFFFFFu - (unsigned)(grp * kTileRows + bi)));
        }
        cons_sync();
        if (tid == kPubThread) {
          __threadfence();
          int old = atom_add_acqrel(p.cnt_lm_done, 1);
          if (old + 1 == p.n_rb_lm) {
            __threadfence();
            // verify steps: draft token j + 1 is accepted while it equals the argmax after
            // position j; the slot keeps the positions up to the last accepted draft
            int acc = 0;
            bool run = p.accepted != nullptr;
            for (int b = 0; b < p.B; ++b) {
              unsigned long long key = atomicExch(p.amax + b, 0ull);
              const int tok = (int)(0xFFFFFFFFu - (unsigned)(key & 0xFFFFFFFFull));
              if (p.next_tokens) p.next_tokens[(size_t)soff * p.rows + b] = tok;
              if (run && b + 1 < p.B && tok == p.tokens[b + 1]) ++acc;
              else run = false;
            }
            if (p.accepted) {
              *p.accepted = acc;
              p.lengths[p.seq0] = m->len[0] + acc + 1;
            }
            atomicExch(p.cnt_lm_done, 0);
            // resident steps: the next step's tokens are written (the release orders them)
            if (p.nsteps > 1) st_release(p.tok_flag, ep);
          }
        }
        break;
      }
    }
  }

  // -------- split-KV GQA attention --------

  // DPL consecutive bf16 values -> fp32 (one 4- or 8-byte load); `l2` for data written by other
  // CTAs in this launch (L2-coherent load), otherwise a plain (shared-memory) load
  template <int DPL>
  __device__ __forceinline__ void load_bf16_row(const uint16_t* src, bool l2, float (&f)[DPL]) {
    if (DPL == 4) {
      uint2 v = l2 ? __ldcg(reinterpret_cast<const uint2*>(src)) : *reinterpret_cast<const uint2*>(src);
      f[0] = bf16lo(v.x);
      f[1] = bf16hi(v.x);
      f[2 % DPL] = bf16lo(v.y);
      f[3 % DPL] = bf16hi(v.y);
    } else {
      uint32_t v = l2 ? __ldcg(reinterpret_cast<const unsigned int*>(src)) : *reinterpret_cast<const uint32_t*>(src);
      f[0] = bf16lo(v);
      f[1 % DPL] = bf16hi(v);
    }
  }

  // Reduce NV partial values across the warp (a butterfly that halves the value count at each
  // level); afterwards lane l holds the total of value index l / (32 / NV).
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

  // Warp 0 waits until every one of n conditions holds: `cond(i)` gives condition i as an
  // address and a value it must reach (unsigned >=; a null address always holds). The lanes
  // write the conditions into a shared table once, then the one out-of-line poller checks them
  // (lane j conditions j, j + 32, ..., one acquire load each), so a wait costs one L2 round trip
  // per poll however many flags it spans. Afterwards the whole CTA agrees on the outcome.
  template <class F>
  __device__ void cta_wait_all(int n, F cond, int where) {
    if (warp == 0) {
      int ok = dead ? 0 : 1;
      if (n > kWaitMax) {  // (no wait of the step spans more: at most max(64 KV heads, 32 row blocks))
        if (lane == 0) raise_err(p, kDevBadArg, 7);
        ok = 0;
      }
      if (ok) {
#pragma unroll 1
        for (int i = lane; i < n; i += 32) {
          const WaitCond c = cond(i);
          m->wt_addr[i] = c.addr;
          m->wt_want[i] = c.want;
        }
        __syncwarp();
        ok = poll_all_geq(m->wt_addr, m->wt_want, n, p.err, p.timeout_ns, where);
      }
      if (lane == 0) m->flag = ok;
    }
    // every consumer thread leaves with the same verdict (one of them may have given up on a
    // ring slot before), so branches on `dead` after a wait are uniform
    dead = cons_any(dead) || !m->flag;
  }

  // a wait condition: a counter reaching target, or a flag reaching a value
  __device__ __forceinline__ WaitCond count_reached(const int* c, int target) const {
    return WaitCond{reinterpret_cast<const unsigned*>(c), (unsigned)target};
  }

  // The unit's q heads, key and value for this token: summed from the published split-K
  // partials, rotated (half-split RoPE at the token's position, angles from the table), rounded
  // to bf16. The unit whose chunk holds the new position also appends k and v to the cache.
  __device__ void qkv_prologue(int l, const AttnUnit& a, float* qkvn) {
    const StageGeo gq = stage_geo(p, K_QKV, 0);
    {
      // the row blocks holding the group's q heads, key and value (at most 6 for head_dim 128)
      const int q0 = a.g * G * HD, k0 = p.hq * HD + a.g * HD, v0 = (p.hq + p.hkv) * HD + a.g * HD;
      const int qa = q0 / kTileRows, qn = (q0 + G * HD - 1) / kTileRows - qa + 1;
      const int ka = k0 / kTileRows, kn = (k0 + HD - 1) / kTileRows - ka + 1;
      const int va = v0 / kTileRows, vn = (v0 + HD - 1) / kTileRows - va + 1;
      const int* cnt = p.cnt_qkv + (size_t)l * p.n_rb_qkv;
      cta_wait_all(qn + kn + vn, [&](int i) {
        const int rb = i < qn ? qa + i : (i < qn + kn ? ka + i - qn : va + i - qn - kn);
        return count_reached(cnt + rb, (int)ep * gq.kbs);
      }, 13);
    }
    // Each thread sums the contributor partials of its NPT values. All loads of a batch of five
    // contributors (for all NPT values, and the thread's RoPE angles) are issued before any is
    // used, so the sums cost one L2 round trip per batch (a q/k/v row block has at most five
    // contributors on 152 SMs); each value is still summed in contributor order.
    constexpr int NV_ = (G + 2) * HD;
    constexpr int NPT = (NV_ + kConsumerWarps * 32 - 1) / (kConsumerWarps * 32);
    float* raw = qkvn + NV_;
    const int pos = m->len[a.b] + soff;
    const size_t pst = (size_t)p.MB * kTileRows;
    const float* pbase[NPT];
    int pnc[NPT], ncmax = 0;
    float psum[NPT];
    float2 cs[NPT];
#pragma unroll
    for (int i = 0; i < NPT; ++i) {
      const int idx = tid + i * kConsumerWarps * 32;
      const int t = idx / HD, d = idx % HD;
      const int row = t < G ? (a.g * G + t) * HD + d : (t == G ? p.hq * HD : (p.hq + p.hkv) * HD) + a.g * HD + d;
      const int rb = row / kTileRows;
      pnc[i] = idx < NV_ ? n_contrib(rb * gq.kbs, gq.kbs, gq.T, gridDim.x) : 0;
      pbase[i] = p.part_qkv + (size_t)rb * gq.kbs * pst + (size_t)a.b * kTileRows + row % kTileRows;
      ncmax = max(ncmax, pnc[i]);
      psum[i] = 0.f;
      cs[i] = (idx < NV_ && t <= G) ? __ldg(p.rope + (size_t)pos * (HD / 2) + d % (HD / 2)) : make_float2(1.f, 0.f);
    }
    for (int c0 = 0; c0 < ncmax; c0 += 5) {
      float v[NPT][5];
#pragma unroll
      for (int i = 0; i < NPT; ++i)
#pragma unroll
        for (int j = 0; j < 5; ++j) v[i][j] = (c0 + j < pnc[i]) ? ldcg(pbase[i] + (size_t)(c0 + j) * pst) : 0.f;
#pragma unroll
      for (int i = 0; i < NPT; ++i)
#pragma unroll
        for (int j = 0; j < 5; ++j) psum[i] += v[i][j];
    }
#pragma unroll
    for (int i = 0; i < NPT; ++i) {
      const int idx = tid + i * kConsumerWarps * 32;
      if (idx < NV_) raw[idx] = psum[i];
    }
    cons_sync();
    const bool writer = (pos / kKvTilePos) >= a.tile0 && (pos / kKvTilePos) < a.tile1;
#pragma unroll
    for (int i = 0; i < NPT; ++i) {
      const int idx = tid + i * kConsumerWarps * 32;
      if (idx >= NV_) break;
      const int t = idx / HD, d = idx % HD;
      float val = raw[idx];
      if (t <= G) {  // q heads and the key rotate; the value does not
        const float other = raw[t * HD + (d < HD / 2 ? d + HD / 2 : d - HD / 2)];
        val = d < HD / 2 ? val * cs[i].x - other * cs[i].y : val * cs[i].x + other * cs[i].y;
      }
      const uint16_t bv = f2bf(val);
      qkvn[idx] = bf16f(bv);
      if (writer && t == G) p.kc[kv_row(p, l, a.b, a.g, pos) + d] = bv;
      if (writer && t == G + 1) p.vc[kv_row(p, l, a.b, a.g, pos) + d] = bv;
    }
    cons_sync();
  }

  // Multi-position steps: the key and value of every new token of the step at KV head a.g, for
  // patching the KV tiles this unit reads (their copies of the cache may predate this step's
  // writes): ext[2j][HD] the key of token j rotated at its position length + j, ext[2j + 1][HD]
  // its value, both rounded to bf16. The sums and the rotation are the prologue's, so the unit's
  // own token comes out bit for bit the same. (The q/k/v counters are complete: waited for by
  // the prologue.)
  __device__ void new_kv_rows(const AttnUnit& a, float* ext) {
    const StageGeo gq = stage_geo(p, K_QKV, 0);
    const size_t pst = (size_t)p.MB * kTileRows;
    const int len0 = m->len[0] + soff;
    constexpr int per = HD / 2 + HD;  // the key's rotation pairs, then the value's elements
    auto sum = [&](int row, int j) {
      const int rb = row / kTileRows;
      const int nc = n_contrib(rb * gq.kbs, gq.kbs, gq.T, gridDim.x);
      const float* src = p.part_qkv + (size_t)rb * gq.kbs * pst + (size_t)j * kTileRows + row % kTileRows;
      float acc = 0.f;
#pragma unroll 1
      for (int c = 0; c < nc; ++c) acc += ldcg(src + (size_t)c * pst);
      return acc;
    };
#pragma unroll 1
    for (int idx = tid; idx < p.B * per; idx += kConsumerWarps * 32) {
      const int j = idx / per, r = idx % per;
      if (r < HD / 2) {
        const int row = p.hq * HD + a.g * HD + r;
        const float x0 = sum(row, j), x1 = sum(row + HD / 2, j);
        const float2 cs = __ldg(p.rope + (size_t)(len0 + j) * (HD / 2) + r);
        ext[(2 * j) * HD + r] = bf16f(f2bf(x0 * cs.x - x1 * cs.y));
        ext[(2 * j) * HD + r + HD / 2] = bf16f(f2bf(x1 * cs.x + x0 * cs.y));
      } else {
        const int d = r - HD / 2;
        ext[(2 * j + 1) * HD + d] = bf16f(f2bf(sum((p.hq + p.hkv) * HD + a.g * HD + d, j)));
      }
    }
    cons_sync();
  }

  // wait for the merged attention output of every (sequence, KV head) whose heads the
  // CTA's output-projection tiles read
  __device__ void wait_o_groups(int l) {
    const StageGeo go = stage_geo(p, K_O, 0);
    const int t0 = range_lo(go.T, blockIdx.x, gridDim.x), t1 = range_lo(go.T, blockIdx.x + 1, gridDim.x);
    // the tiles' k blocks (input columns) kb_a .. kb_b, wrapping at kbs, all of them when the
    // range spans a whole row block; k block kb reads the heads of groups grp_lo(kb) .. grp_hi(kb)
    auto grp_lo = [&](int kb) { return kb * kTileK / HD / G; };
    auto grp_hi = [&](int kb) { return ((kb + 1) * kTileK - 1) / HD / G; };
    auto bits = [](int lo, int hi) { return (2ull << hi) - (1ull << lo); };  // bits lo..hi, hi <= 63
    unsigned long long mask = 0;
    if (t1 > t0) {
      const int kb_a = t0 % go.kbs, kb_b = (t1 - 1) % go.kbs;
      if (t1 - t0 >= go.kbs)
        mask = bits(0, grp_hi(go.kbs - 1));
      else if (kb_a <= kb_b)
        mask = bits(grp_lo(kb_a), grp_hi(kb_b));
      else
        mask = bits(grp_lo(kb_a), grp_hi(go.kbs - 1)) | bits(0, grp_hi(kb_b));
    }
    // condition g = KV head g's merged slices of every sequence (B * nch of them) for the flagged
    // heads; unflagged heads pass at once
    const int* f = p.o_cnt + (size_t)l * p.hkv;
    cta_wait_all(p.hkv, [&](int g) {
      return ((mask >> g) & 1ull) ? count_reached(f + g, p.B * p.nch) : WaitCond{nullptr, 0u};
    }, 16);
  }

  // wait for the final SwiGLU rows of the n experts whose down-projection k blocks the CTA's
  // tiles read: expert slots v0, v0 + 1, ... (wrapping after nv; slot U is the shared expert)
  __device__ void wait_h(int l, int v0, int n, int nv, int U) {
    cta_wait_all(n, [&](int j) {
      const int v = (v0 + j) % nv;
      const int slot = v < U ? v : p.umax;
      return count_reached(p.h_cnt + (size_t)l * (p.umax + 1) + slot, (int)ep * p.n_rb_gu);
    }, 17);
  }

  __device__ void attn_stage(int l) {
    constexpr int DPL = HD / 32;       // dims per lane
    constexpr int PPW = kKvTilePos / kConsumerWarps;  // positions per warp in a KV tile (8)
    static_assert(2 * kKvTilePos * HD * 2 <= kSlotBytes, "a KV tile (K and V rows) must fit one slot");
    constexpr int NV = PPW * G;                        // scores per warp per tile
    static_assert(NV <= 32 && (NV & (NV - 1)) == 0, "scores per warp must be a power of two <= 32");
    constexpr int LPV = 32 / NV;                       // lanes holding each reduced score
    static_assert(DPL == 2 || DPL == 4, "head_dim 64 or 128");
    const float qscale = 1.4426950408889634f / sqrtf((float)HD);  // log2(e)/sqrt(hd)
    const unsigned row_bytes = HD * 2;
    const int NU = p.B * p.hkv * p.nch;
    trace(7 << 4);
    for (int u = blockIdx.x; u < NU; u += gridDim.x) {
      AttnUnit a = attn_unit(p, m, u, soff);
      // The group's q heads, k and v for this token, rotated and rounded to bf16, in shared
      // memory: qkvn[t][HD] with t < G the query heads, t = G the key, t = G + 1 the value.
      float* qkvn = red;
      if (a.tile1 > a.tile0) qkv_prologue(l, a, qkvn);
      // multi-position steps: the unit's tiles hold some of the step's new positions
      float* ext = qkvn + 2 * (G + 2) * HD;
      const bool mnew = p.mpos && a.tile1 > a.tile0 && (m->len[0] + soff + p.B - 1) / kKvTilePos >= a.tile0 &&
                        (m->len[0] + soff) / kKvTilePos < a.tile1;
      if (mnew) new_kv_rows(a, ext);
      float q[G][DPL];
#pragma unroll
      for (int h = 0; h < G; ++h)
#pragma unroll
        for (int j = 0; j < DPL; ++j) q[h][j] = qkvn[h * HD + lane * DPL + j] * qscale;
      float mrun[G], lrun[G], acc[G][DPL];
#pragma unroll
      for (int h = 0; h < G; ++h) {
        mrun[h] = -INFINITY;
        lrun[h] = 0.f;
#pragma unroll
        for (int j = 0; j < DPL; ++j) acc[h][j] = 0.f;
      }
      const int newpos = a.T - 1;
      const int vidx = lane / LPV;
      const int my_i = vidx / G, my_h = vidx % G;  // the (position, head) score this lane ends with
      // All eight warps share each KV tile; warp w takes positions 4w..4w+3 and keeps its own
      // online-softmax state (merged across warps after the unit's last tile).
      for (int t = a.tile0; t < a.tile1; ++t) {
        const uint8_t* slot = wait_item();
        {
          // This step's key and value (from the prologue; the slot's copy of the cache may predate
          // them) are written into the slot once, so the loops below read every position alike.
          const int jn = newpos - t * kKvTilePos;
          if (p.mpos) {
            // every new position up to the unit's own (causal) that falls in this tile
            if (mnew) {
              const int first = m->len[0] + soff - t * kKvTilePos;
              bool hit = false;
#pragma unroll 1
              for (int jj = 0; jj <= a.b; ++jj) {
                const int r = first + jj;
                if (r < 0 || r >= kKvTilePos) continue;
                hit = true;
                uint16_t* kr = reinterpret_cast<uint16_t*>(const_cast<uint8_t*>(slot) + r * row_bytes);
                uint16_t* vr = reinterpret_cast<uint16_t*>(const_cast<uint8_t*>(slot) + (kKvTilePos + r) * row_bytes);
                if (!dead)
                  for (int d = tid; d < HD; d += kConsumerWarps * 32) {
                    kr[d] = f2bf(ext[(2 * jj) * HD + d]);
                    vr[d] = f2bf(ext[(2 * jj + 1) * HD + d]);
                  }
              }
              if (hit) cons_sync();  // (the same for all warps)
            }
          } else if (jn >= 0 && jn < kKvTilePos) {  // the same for all warps (`dead` may not be)
            uint16_t* kr = reinterpret_cast<uint16_t*>(const_cast<uint8_t*>(slot) + jn * row_bytes);
            uint16_t* vr = reinterpret_cast<uint16_t*>(const_cast<uint8_t*>(slot) + (kKvTilePos + jn) * row_bytes);
            if (!dead)
              for (int d = tid; d < HD; d += kConsumerWarps * 32) {
                kr[d] = f2bf(qkvn[G * HD + d]);
                vr[d] = f2bf(qkvn[(G + 1) * HD + d]);
              }
            cons_sync();
          }
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
              load_bf16_row<DPL>(reinterpret_cast<const uint16_t*>(slot + j * row_bytes) + lane * DPL, false, kf);
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
          // per-head maximum over this warp's positions (value-index bits above log2(G))
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
              float vf[DPL];
              load_bf16_row<DPL>(reinterpret_cast<const uint16_t*>(slot + (kKvTilePos + j) * row_bytes) + lane * DPL,
                                 false, vf);
#pragma unroll
              for (int h = 0; h < G; ++h)
#pragma unroll
                for (int d = 0; d < DPL; ++d) acc[h][d] = fmaf(pv[i * G + h], vf[d], acc[h][d]);
            }
          }
        }
        release_item();
      }
      cons_sync();
      trace(7 << 4 | 1);
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
      // publish: the CTA barrier orders every thread's partial before the publishing thread's
      // releasing arrival (the layer's counters start the launch at zero, see stage_rmsnorm)
      cons_sync();
      const size_t gi = ((size_t)l * p.MB + a.b) * p.hkv + a.g;
      if (tid == kPubThread && !dead) red_release_add(p.attn_cnt + gi, 1);
      // Chunk merge, shared by the group's nch units (with nch > 1 the host makes every unit a
      // CTA of its own, so a CTA waits only for others' chunks): unit c merges the outputs
      // [o_lo, o_hi) = [c * G*HD / nch, (c+1) * G*HD / nch) of the group's G*HD (head o / HD, dim
      // o % HD) once every chunk has arrived, and arrives on the group's merged counter. Weights
      // per head h: w_c = exp2(m_c - M) / L with M = max_c m_c, L = sum_c exp2(m_c - M) l_c (warp
      // h - h_lo reduces them over the chunks, in a fixed order); output o = sum_c w_c acc_c[o],
      // in chunk order.
      cta_wait_all(1, [&](int) { return count_reached(p.attn_cnt + gi, p.nch); }, 23);
      if (!dead) {  // (uniform across the CTA after a wait)
        constexpr int kMergeBatch = 24;
        const int o_lo = range_lo(G * HD, a.c, p.nch), o_hi = range_lo(G * HD, a.c + 1, p.nch);
        const int h_lo = o_lo / HD, nh = o_hi > o_lo ? (o_hi - 1) / HD - h_lo + 1 : 0;
        const float* src = p.attn_part + ((size_t)a.b * p.hkv + a.g) * p.nch * G * (HD + 2);
        const size_t cst = (size_t)G * (HD + 2);  // chunk stride
        float* cw = red;                          // [nh][nch] weights
        // the first output of this thread: its chunk values are loaded before the weights are
        // formed, all in flight together (one pass covers the slice unless nch is tiny)
        int o = o_lo + tid;
        const float* vsrc = src + (size_t)(o / HD) * (HD + 2) + o % HD;
        float mv[kMergeBatch];
#pragma unroll
        for (int j = 0; j < kMergeBatch; ++j) mv[j] = (o < o_hi && j < p.nch) ? ldcg(vsrc + (size_t)j * cst) : 0.f;
#pragma unroll 1
        for (int hh = warp; hh < nh; hh += kConsumerWarps) {
          const float* ms = src + (size_t)(h_lo + hh) * (HD + 2) + HD;  // (m, l) of chunk 0
          float mx = -INFINITY;
#pragma unroll 1
          for (int c = lane; c < p.nch; c += 32) mx = fmaxf(mx, ldcg(ms + (size_t)c * cst));
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
          float ls = 0.f;
#pragma unroll 1
          for (int c = lane; c < p.nch; c += 32) {
            const float mc = ldcg(ms + (size_t)c * cst);
            if (mc != -INFINITY) ls = fmaf(exp2f(mc - mx), ldcg(ms + (size_t)c * cst + 1), ls);
          }
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) ls += __shfl_xor_sync(0xffffffffu, ls, off);
#pragma unroll 1
          for (int c = lane; c < p.nch; c += 32) {
            const float mc = ldcg(ms + (size_t)c * cst);
            cw[hh * p.nch + c] = (mc == -INFINITY || !(ls > 0.f)) ? 0.f : exp2f(mc - mx) / ls;
          }
        }
        cons_sync();
#pragma unroll 1
        for (; o < o_hi; o += kConsumerWarps * 32) {
          if (o != o_lo + tid) {
            vsrc = src + (size_t)(o / HD) * (HD + 2) + o % HD;
#pragma unroll
            for (int j = 0; j < kMergeBatch; ++j) mv[j] = j < p.nch ? ldcg(vsrc + (size_t)j * cst) : 0.f;
          }
          const float* w = cw + (o / HD - h_lo) * p.nch;
          float A = 0.f;
#pragma unroll
          for (int j = 0; j < kMergeBatch; ++j)
            if (j < p.nch) A = fmaf(w[j], mv[j], A);
#pragma unroll 1
          for (int c = kMergeBatch; c < p.nch; ++c)  // more chunks than one batch (small models)
            A = fmaf(w[c], ldcg(vsrc + (size_t)c * cst), A);
          p.obuf[(size_t)a.b * p.hq * HD + (size_t)a.g * G * HD + o] = f2bf(A);
        }
        cons_sync();
        if (tid == kPubThread) red_release_add(p.o_cnt + (size_t)l * p.hkv + a.g, 1);
      }
      cons_sync();
    }
    trace(7 << 4 | 2);
  }

  // -------- the step --------

  // The step: per layer a fixed sequence of phases, each ending in at most one GEMV stage; then
  // the final norm and the LM head. Every GEMV stage goes through the one gemv_stage call below,
  // so its code (the hot tile loop, flushes and finalisers) exists once in the kernel: the
  // instruction working set of a layer then stays small enough to be cached.
  __device__ void run() {
    trace(10 << 4);
    if (blockIdx.x == 0 && tid == 0) p.layer_ts[0] = gtimer();
    // the TMEM accumulators of the tensor-core tiles (warp 0 allocates and frees them)
    if constexpr (kTC) {
      if (warp == 0) tmem_alloc(&m->tmem_base, kTmemCols);
      tc_fence_before();
      cons_sync();
      tc_fence_after();
      tmem = m->tmem_base;
    }
    int U = 0;
#pragma unroll 1
    for (soff = 0; soff < p.nsteps; ++soff) {
    ep = p.epoch + (unsigned)soff;
    if (soff > 0) {
      // resident steps: this step's tokens are the previous step's argmax (its last LM finaliser
      // publishes the flag after writing them)
      cta_wait_all(1, [&](int) { return WaitCond{p.tok_flag, ep - 1u}; }, 26);
      if (tid < p.B) {
        int tok = __ldcg(p.tokens + (size_t)soff * p.rows + tid);
        if (tok < 0 || tok >= p.V) {
          raise_err(p, kDevBadArg, 2);
          tok = 0;
        }
        m->tok[tid] = tok;
      }
      cons_sync();
    }
#pragma unroll 1
    for (int l = 0; l <= p.L; ++l) {
      const bool lm = l == p.L;
      if (lm && p.V == 0) break;
#pragma unroll 1
      for (int ph = 0; ph < 7; ++ph) {
        int kind = -1;
        // a norm stage or an activation copy runs right before the GEMV stage it feeds (one call
        // site each, see below): the attention output, or the SwiGLU rows of cp_n experts
        const uint16_t* norm_w = nullptr;
        bool norm_from_o = false;
        int cp_v0 = 0, cp_n = 0, cp_nv = 1;  // experts cp_v0, cp_v0 + 1, ... (mod cp_nv)
        bool cp_obuf = false;
        if (lm) {
          if (ph == 0) {
            norm_w = p.final_norm;
            kind = K_LM;
          }
        } else {
          const LayerDev& Ld = p.layers[l];
          switch (ph) {
            case 0:
              // attention block: q/k/v partials -> attention units (wait on their row blocks) ->
              // merged head outputs -> output projection (waits on the groups it reads)
              norm_w = Ld.attn_norm;
              kind = K_QKV;
              break;
            case 1:
              cta_stamp(l, S_QKV_DONE);
              attn_stage(l);
              cta_stamp(l, S_ATTN_DONE);
              wait_o_groups(l);
              cta_stamp(l, S_OGRP_READY);
              cp_obuf = true;
              cp_n = 1;
              kind = K_O;
              break;
            case 2:
              cta_stamp(l, S_O_DONE);
              // FFN block: x_mid from the projection partials (waits on every row block)
              norm_w = Ld.ffn_norm;
              norm_from_o = true;
              U = 0;
              kind = p.dense ? K_SHGU : K_ROUTER;
              break;
            case 3:
              if (!p.dense) {
                cta_stamp(l, S_FFN_PRE_DONE);
                local_routing(l);
                trace(9 << 4);
                U = m->U;
                cta_stamp(l, S_ROUTED);
                if (p.nsh) kind = K_SHGU;
              }
              break;
            case 4:
              if (!p.dense) kind = K_RTGU;
              break;
            case 5: {
              cta_stamp(l, S_GU_DONE);
              // down projections of all active experts, gate-weighted, + residual
              // (the CTA's tiles run through expert runs s0 .. s1 of tpe tiles, run s of expert
              // slot s % nv: it stages the SwiGLU rows of the first min(runs, nv) of them)
              const StageGeo g = stage_geo(p, K_D, U);
              const int t0 = range_lo(g.T, blockIdx.x, gridDim.x), t1 = range_lo(g.T, blockIdx.x + 1, gridDim.x);
              const int nv = U + p.nsh;
              int s0 = 0, nst = 0;
              if (t1 > t0) {
                s0 = t0 / g.tpe;
                nst = min((t1 - 1) / g.tpe - s0 + 1, nv);
              }
              if (nst * p.inter > p.xmax) {
                raise_err(p, kDevBadArg, 6);
                nst = 0;
              }
              const int v0 = nv > 0 ? s0 % nv : 0;
              wait_h(l, v0, nst, nv, U);
              cta_stamp(l, S_H_READY);
              for (int i = tid; i < BM; i += 256) m->gate[i][U] = 1.f;  // shared / dense expert
              cp_v0 = v0;
              cp_n = nst;
              cp_nv = nv;
              kind = K_D;
              break;
            }
            default:
              cta_stamp(l, S_D_DONE);
              // no grid barrier: the next layer's norm waits for the output row blocks it reads,
              // and every buffer a later stage overwrites is read before an all-to-all exchange
              // that the overwriting stage depends on
              trace(8 << 4 | 1);
              cta_stamp(l, S_BARRIER);
              if (l == 0 && blockIdx.x == 0 && tid == 0 && !dead)
                for (int b = 0; b < p.B; ++b) p.lengths[p.mpos ? p.seq0 : p.seq0 + b] = m->len[b] + soff + 1;
              break;
          }
        }
        if (norm_w) {
          stage_rmsnorm(lm ? p.L : l, nullptr, norm_w, norm_from_o);
          if (norm_from_o) cta_stamp(l, S_XMID_READY);
        }
        if (cp_n > 0) {
          int v = cp_v0;
#pragma unroll 1
          for (int j = 0; j < cp_n; ++j) {
            const uint16_t* src = cp_obuf ? p.obuf : (v < U ? p.hrt + (size_t)v * p.MB * p.inter : p.hsh);
            const int n = cp_obuf ? p.hq * HD : p.inter;
            stage_copy(src, n, (size_t)n, j * n);
            if (++v == cp_nv) v = 0;
          }
          cons_sync();
        }
        if (kind >= 0) gemv_stage(kind, lm ? 0 : l, lm ? 0 : U);
      }
    }
    }
    trace(10 << 4 | 1);
    if (blockIdx.x == 0 && tid == 0) p.layer_ts[p.L + 1] = gtimer();
    // Free TMEM once the MMA warp has finished (it waits for its last MMAs before saying so);
    // the wait is bounded whatever the status word says.
    if (kTC && warp == 0) {
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
// MMA warp: one thread walks the CTA's GEMV tiles in the consumers' order and hands each to the
// tensor cores once its ring slot has landed, its stage's activations are staged and its group
// of TMEM slices is free, up to kNG groups ahead of the consumers.

template <int BM, int HD, int G>
struct MmaIssuer {
  const KParams& p;
  uint8_t* ring;
  uint64_t* full;
  uint64_t* mempty;
  Misc* m;
  const uint8_t* xsb;  // the B operand region
  int slot = 0;        // ring slot of the next item (items: GEMV slots and the attention's KV tiles)
  unsigned lap = 0;
  unsigned gseq = 0, stage = 0;
  bool dead = false;
  uint32_t tmem = 0;
  BGeo bg;
  int soff = 0;      // resident steps done in this launch
  unsigned lay = 0;  // layers done in this launch (the routing barrier's phase)

  __device__ MmaIssuer(const KParams& p_, uint8_t* r, uint64_t* f, uint64_t* me, Misc* m_, const uint8_t* x)
      : p(p_), ring(r), full(f), mempty(me), m(m_), xsb(x) {
    bg = bgeo(p.B);
  }

  __device__ __forceinline__ void skip(int n) {
    for (int i = 0; i < n; ++i)
      if (++slot == p.ring) {
        slot = 0;
        ++lap;
      }
  }

  // The stage's tiles in groups of up to kGT per segment (as the consumers take them): each tile
  // gets TMEM slice (group slot) * kGT + i; a slot is freed (commit on its mempty barrier) after
  // its last tile's MMAs, a group announced (commit on tfull) after its last tile's.
  // wait (bounded) until the consumers have staged the operand of GEMV stage number `stage`
  __device__ void wait_staged() {
    if (dead) return;
    const unsigned long long t0 = gtimer();
    for (unsigned it = 1; *reinterpret_cast<volatile unsigned*>(&m->stages_staged) < stage; ++it) {
      if ((it & 63u) == 0) {
        if (aborted(p)) {
          dead = true;
          return;
        }
        if (gtimer() - t0 > p.timeout_ns) {
          raise_err(p, kDevTimeout, 26);
          dead = true;
          return;
        }
      }
    }
    __threadfence_block();
  }

  __device__ void gemv(int kind, int U) {
    ++stage;
    wait_staged();
    tc_fence_after();
    tmem = m->tmem_base;
    const StageGeo g = stage_geo(p, kind, U);
    const int t0 = range_lo(g.T, blockIdx.x, gridDim.x), t1 = range_lo(g.T, blockIdx.x + 1, gridDim.x);
    const int nv = kind == K_D ? U + p.nsh : 1;
    TilePos pos;
    pos.init(p, g, kind, t0, t1);
    constexpr uint32_t idesc = idesc_e4m3_f32(kTileRows, kMmaN);
    const uint32_t sbo = bg.nrb == 16 ? 1024u : 0u;  // 8-row blocks: the second row group aliases the first
    int j = 0;
#pragma unroll 1
    for (int t = t0; t < t1;) {
      const int n = min(kGT, min(t1, (pos.seg + 1) * g.kbs) - t);
      const int gsl = gseq % kNG;
      if (!dead && gseq >= (unsigned)kNG && !mbar_wait(&m->tempty[gsl], (gseq / kNG - 1) & 1, p, 28)) dead = true;
#pragma unroll 1
      for (int i = 0; i < n; ++i, ++t) {
        if (!dead && j == 0 && !mbar_wait(&full[slot], lap & 1, p, 27)) dead = true;
        const uint8_t* a = ring + (size_t)slot * kSlotBytes + (size_t)j * kTileBytes;
        if (!dead) {
          tc_fence_after();
          m->hdr[gsl][i] = *reinterpret_cast<const float2*>(a + kTileData);
          const int kbi = pos.kbi(p, kind);
          const uint8_t* b = xsb + (size_t)(kbi / bg.pk) * bg.nrb * 128;
          const uint64_t ad = smem_desc(a, 128, 1024), bd = smem_desc(b, 128, sbo);
          const uint32_t d = tmem + (uint32_t)((gsl * kGT + i) * kMmaN);
#pragma unroll
          for (int k = 0; k < kTileK / 32; ++k)  // 32 bytes of K per MMA: two core matrices (256 B)
            mma_e4m3(d, ad + (uint64_t)(k * 16), bd + (uint64_t)(k * 16), idesc, k > 0 ? 1u : 0u);
        }
        pos.next(p, g, kind, nv);
        if (++j == kSlotTiles || t == t1 - 1) {
          if (!dead) mma_commit(&mempty[slot]);  // the slot's tiles are read once these MMAs are done
          j = 0;
          skip(1);
        }
      }
      if (!dead) {
        // the group's products are ready once both arrivals are in: the commit (MMAs done) and
        // this thread's own (a release that orders its header copies before the consumers' reads)
        mma_commit(&m->tfull[gsl]);
        mbar_arrive(&m->tfull[gsl]);
      }
      ++gseq;
    }
  }

  // the same stage sequence as the consumers (and the producer): per layer q/k/v, attention (its
  // KV tiles pass through the ring), output projection, router or dense FFN, routing, shared
  // expert, routed gate/up, down projections; then the LM head
  __device__ void run() {
#pragma unroll 1
    for (soff = 0; soff < p.nsteps; ++soff)
#pragma unroll 1
    for (int l = 0; l <= p.L; ++l) {
      if (l == p.L) {
        if (p.V > 0) gemv(K_LM, 0);
        break;
      }
      gemv(K_QKV, 0);
      int items = 0;
      for (int u = blockIdx.x; u < p.B * p.hkv * p.nch; u += gridDim.x) {
        const AttnUnit a = attn_unit(p, m, u, soff);
        items += a.tile1 - a.tile0;
      }
      skip(items);
      gemv(K_O, 0);
      int U = 0;
      if (p.dense) {
        gemv(K_SHGU, 0);
      } else {
        gemv(K_ROUTER, 0);
        if (!dead && !mbar_wait(&m->rt_bar, lay & 1u, p, 29)) dead = true;
        U = min(max(m->U, 0), p.umax);
        if (p.nsh) gemv(K_SHGU, 0);
        gemv(K_RTGU, U);
      }
      gemv(K_D, U);
      ++lay;
    }
    // the last MMAs complete before the consumers may free TMEM (bounded wait)
    if (gseq > 0) {
      const unsigned last = gseq - 1;
      const unsigned long long t0 = gtimer();
      while (!mbar_try_wait(&m->tfull[last % kNG], (last / kNG) & 1) && gtimer() - t0 < p.timeout_ns) {
      }
    }
    mbar_arrive(&m->mma_done);
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
  uint64_t* mempty = reinterpret_cast<uint64_t*>(smem + L.mempty_off);
  uint16_t* xs = reinterpret_cast<uint16_t*>(smem + L.xs_off);
  float* red = reinterpret_cast<float*>(smem + L.red_off);
  Misc* m = reinterpret_cast<Misc*>(smem + L.misc_off);

  const int tid = threadIdx.x;
  if (tid == 0) {
    for (int s = 0; s < p.ring; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
      mbar_init(&mempty[s], 1);
    }
    mbar_init(&m->rt_bar, 1);
    m->stages_staged = 0;
    mbar_init(&m->mma_done, 1);
    for (int i = 0; i < kNG; ++i) {
      mbar_init(&m->tfull[i], 2);  // MMA commit + the MMA thread's release of the headers
      mbar_init(&m->tempty[i], kConsumerWarps);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // the B operand region starts zero: rows beyond the step's tokens are never written
  for (int i = tid; i < (L.red_off - L.xs_off) / 16; i += kThreads)
    reinterpret_cast<uint4*>(smem + L.xs_off)[i] = make_uint4(0u, 0u, 0u, 0u);
  if (tid < kMaxBatch) {
    int len = 0, tok = 0;
    if (tid < p.B) {
      len = p.mpos ? p.lengths[p.seq0] + tid : p.lengths[p.seq0 + tid];
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
      Producer<BM, HD, G> prod(p, ring, full, empty, mempty, m);
      prod.run();
    } else if (BM >= 2 && tid == (kConsumerWarps + 1) * 32) {  // (tensor-core tiles: steps of 2+ tokens)
      MmaIssuer<BM, HD, G> mma(p, ring, full, mempty, m, smem + L.xs_off);
      mma.run();
    }
    return;
  }
  Consumer<BM, HD, G> cons(p, ring, full, empty, xs, red, m);
  cons.run();
}

}  // namespace dec
