// The decode step for 5 .. 64 tokens (sequences side by side): the tensor-core expert GEMMs of a
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
// write one split-K partial per output row block. A routed expert's tiles multiply only its own
// tokens: after the routing every CTA knows each expert slot's tokens, their B rows are gathered
// into compact blocks (the slot's j-th token in rows 2j, 2j + 1), and the MMA's N is twice the
// slot's token count rounded up to 16. Attention runs on the tensor cores too (bf16 K q^T and
// V^T P per 64-position KV tile, the tile loaded by tensor-map copies in the layout the MMAs read).
//
// Phases of a layer (barrier after each):
//   q/k/v GEMV | attention (each unit sums its q/k/v partials, applies RoPE, appends its key and
//   value, streams its KV tiles) | chunk merge -> B blocks of the attention output | output
//   projection GEMV | x_mid = x + projection, RMSNorm -> B blocks | router and shared expert
//   gate/up GEMVs | routing (one CTA per token) | each slot's tokens' B rows gathered | routed
//   gate/up GEMV | SwiGLU -> B blocks per expert slot | down GEMV (expert-major, gate applied per
//   partial) | layer output, next RMSNorm -> B blocks.
// Then the LM head GEMV, its finalisation (logits, argmax) and the next tokens.
#pragma once
#include "dec_kernel.cuh"

namespace dec {
namespace wide {

constexpr int kGC = 256;           // TMEM columns per group of tile products
constexpr int kNGW = 2;            // groups in flight (all 512 columns)
constexpr int kBarsPerLayer = 12;  // grid barriers of one layer
constexpr int kWideTopk = 8;       // experts per token the wide kernel's routing tables hold
// diagnostics build: CTA 0's wait totals (ns) over the step's routed gate/up stages, in trace
// words kWaitTrace + {0: producer waiting for copies in flight, 1: producer waiting for slot
// releases, 2: MMA waiting for slot data, 3: MMA waiting for free TMEM, 4: consumers waiting for
// products, 5: consumers' stage time}
constexpr int kWaitTrace = 400;

// Ring slot: two weight tiles and an 8 KB B area. Two tiles whose B blocks fit half the area each
// (up to 32 rows, 16 tokens) share a slot, their blocks side by side (a 32 KB weight hand-off;
// one SM's streaming rate grows with the bytes per hand-off up to ~32 KB). A wider tile (a dense
// stage of more than 16 tokens, an expert with more) has a slot to itself, its block in the
// second tile's place. Four slots fit beside the GEMV accumulators (below).
__host__ __device__ constexpr int b_area(int) { return 8192; }
__host__ __device__ constexpr int pair_rows(int nr) { return b_area(nr) / 2 / 128; }
__host__ __device__ constexpr int slot_bytes(int nr) { return 2 * kTileBytes + b_area(nr); }

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
  // expert stages split by work (see wsplit below): prefix sums of the slots' tile weights, or
  // null for the even split by tiles; WT = the stage's total weight (WT x grid < 2^32, checked
  // by the host)
  const int* pw;
  unsigned WT;
};
// Routed gate/up: U expert slots x n_rb_gu row blocks x kb_d k blocks. Down: U + n_shared slots
// (the shared expert last), expert major, segment (u, rb) = its kb_i k blocks.
__host__ __device__ inline WGeo wgeo(const KParams& p, int kind, int U, int G) {
  WGeo g;
  g.tpe = 0;
  g.pw = nullptr;
  g.WT = 0;
  switch (kind) {
    case K_QKV: g.kbs = p.kb_d; g.T = p.n_rb_qkv * p.kb_d; break;
    case K_O: g.kbs = p.kb_o; g.T = p.n_rb_d * p.kb_o; break;
    case K_ROUTER: g.kbs = p.kb_d; g.T = p.n_rb_router * p.kb_d; break;
    case K_SHGU: g.kbs = p.kb_d; g.T = p.n_rb_gu * p.kb_d; break;
    case K_RTGU: g.kbs = p.kb_d; g.tpe = p.n_rb_gu * p.kb_d; g.T = U * g.tpe; break;
    case K_D: g.kbs = p.kb_i; g.tpe = p.n_rb_d * p.kb_i; g.T = (U + p.nsh) * g.tpe; break;
    default: g.kbs = p.kb_d; g.T = p.n_rb_lm * p.kb_d; break;
  }
  // expert stages: one slot per k block (any split, even or by work, fits)
  g.S = (kind == K_RTGU || kind == K_D) ? g.kbs : seg_slots(g.T, g.kbs, G);
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
  int pw[kMaxExperts + 2];                    // prefix sums of the slots' tile weights (wsplit)
  int wmax;                                   // the heaviest slot's weight
  alignas(8) uint8_t wsel[kWideMax][kWideTopk];  // expert slot of each token's selections
  float wgate[kWideMax][kWideTopk];           // and their gates
  float rsum[kConsumerWarps];
  // attention on the tensor cores: the consumers' own MMA completions, and per tile the two
  // position warps' score maxima, the rescale factors and, per unit, the softmax state per head
  uint64_t sbar, obar;  // a round's S^T and O^T products done
  float amx[4][8], acr[8], alw[4][8], amr[8];
  alignas(16) int8_t ex[kMaxKb * kWideMax];  // exponents of the running GEMV stage's B blocks [row][token]
};

// Work-weighted split of an expert stage. A tile of expert slot u costs w(u) = its B rows / 16
// (at least 2): the epilogue work and the slot pairing grow with the slot's tokens, and at large
// batches one slot (the shared expert's, or a routed one that drew many tokens) can cost several
// times the rest. Tile t of slot u starts at weight position tpe pw[u] + (t - u tpe) w(u); CTA c
// owns the tiles whose start lies in [c WT / G, (c + 1) WT / G), a contiguous range. Used when
// a CTA's share WT / G is at least the heaviest tile (so every CTA owns a tile of each segment it
// straddles); otherwise, and whenever the stage has fewer tiles than CTAs, the even split.
__device__ __forceinline__ unsigned wpos(const WGeo& g, int t) {
  const int u = t / g.tpe;
  return (unsigned)(g.tpe * g.pw[u] + (t - u * g.tpe) * (g.pw[u + 1] - g.pw[u]));
}
__device__ __forceinline__ int wowner(const WGeo& g, int t, int G) { return (int)(wpos(g, t) * (unsigned)G / g.WT); }
// first tile of CTA c (c = G: the stage's end)
__device__ inline int wstart(const WGeo& g, int c, int G) {
  if (!g.pw) return range_lo(g.T, c, G);
  if (c >= G) return g.T;
  const unsigned P = ((unsigned)c * g.WT + (unsigned)G - 1u) / (unsigned)G;
  int u = 0;
  while ((unsigned)(g.tpe * g.pw[u + 1]) <= P) ++u;
  const unsigned r = P - (unsigned)(g.tpe * g.pw[u]);
  const unsigned w = (unsigned)(g.pw[u + 1] - g.pw[u]);
  return u * g.tpe + (int)min((unsigned)g.tpe, (r + w - 1u) / w);
}
// contributors of segment seg, and CTA c's slot among them (its first tile of the segment: f)
__device__ __forceinline__ int wn_contrib(const WGeo& g, int seg, int G) {
  if (!g.pw) return n_contrib(seg * g.kbs, g.kbs, g.T, G);
  return wowner(g, seg * g.kbs + g.kbs - 1, G) - wowner(g, seg * g.kbs, G) + 1;
}
__device__ __forceinline__ int wcontrib_slot(const WGeo& g, int c, int f, int seg, int G) {
  if (!g.pw) return contrib_slot(c, f, seg * g.kbs, g.T, G);
  return c - wowner(g, seg * g.kbs, G);
}

// attach the work-weighted split to an expert stage's geometry where it applies (the slots'
// weights come from the CTA's routing tables)
template <class M>
__device__ __forceinline__ void wsplit(WGeo& g, const M* m, const KParams& p, int kind, int U, int G) {
  if ((kind != K_RTGU && kind != K_D) || g.T < G) return;
  const unsigned WT = (unsigned)(g.tpe * m->pw[kind == K_RTGU ? U : U + p.nsh]);
  if (WT / (unsigned)G < (unsigned)m->wmax) return;
  g.pw = m->pw;
  g.WT = WT;
}

struct WLayout {
  int ring_off, full_off, empty_off, mempty_off, red_off, acc_off, misc_off, total;
};
// Attention operands staged by the consumers (att_* offsets, whole 128-byte core matrices): the
// probabilities P as [position block][column][8 positions] (16 columns) and the group's query
// heads as [d chunk][head row][8 values] (16 rows). K and V stay in their ring slot.
__host__ __device__ constexpr int att_p(int) { return 0; }
__host__ __device__ constexpr int att_q(int) { return 2 * kKvTilePos * 16 * 2; }  // (P: two tiles)
__host__ __device__ constexpr int att_bytes(int hd) { return att_q(hd) + 16 * hd * 2; }

// The K (or V) of a round of two KV tiles in a ring slot: from the first 1024-byte boundary,
// head_dim / 64 parts of 128 positions x 128 bytes in the 128-byte swizzled layout (part b: d =
// 64 b .. 64 b + 63), each filled by two 64 x 64 boxes
__device__ __forceinline__ uint8_t* kv_area(uint8_t* slot) {
  return slot + ((1024u - (smem_u32(slot) & 1023u)) & 1023u);
}
// The GEMV accumulators live in shared memory, not registers: nr / 4 per consumer thread (up to
// 32) did not fit beside the rest of the kernel's live state at the 168-register cap, and the
// spills cost more than the shared-memory round trips (measured: 64 tokens 13761 vs 11452
// tokens/s, 16 tokens 6144 vs 5894).
__host__ __device__ inline WLayout wlayout(int ring, int nr, int hd, int group) {
  WLayout s;
  s.ring_off = 0;
  s.full_off = align_up(ring * slot_bytes(nr), 128);
  s.empty_off = s.full_off + ring * 8;
  s.mempty_off = s.empty_off + ring * 8;
  s.red_off = align_up(s.mempty_off + ring * 8, 128);
  int red = kConsumerWarps * group * (hd + 2) * 4;       // attention: the warps' states
  red = red > 2 * (group + 2) * hd * 4 ? red : 2 * (group + 2) * hd * 4;  // the unit's q/k/v
  // routing marks, SwiGLU pairs, each expert slot's tokens
  const int pairs = (kMaxExperts + kWideMax * 17) * 4 + (kMaxExperts + 1) * kWideMax;
  red = red > pairs ? red : pairs;
  s.acc_off = align_up(s.red_off + red, 128);
  // one float4 per (token chunk, warp half, weight row): thread (row, half) owns its entries; the
  // attention's staging shares the area (no GEMV runs meanwhile)
  int acc = kTileRows * (nr / 2) * 4;
  acc = acc > att_bytes(hd) ? acc : att_bytes(hd);
  s.misc_off = align_up(s.acc_off + acc, 128);
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

// B rows (tokens x 2 pieces, padded to the MMA's N granularity of 16) of n tokens
__device__ __forceinline__ int brows(int n) { return (2 * n + 15) & ~15; }

// tokens a GEMV tile multiplies: its expert slot's (routed stages), or the whole step's
__device__ __forceinline__ int tile_tokens(const KParams& p, const WMisc* m, int kind, const WGeo& g, int t) {
  if (kind == K_RTGU || kind == K_D) return __popcll(m->umask[t / g.tpe]);
  return p.B;
}

// TMEM columns of one tile's product (its B rows) and tiles per group (one hand-off between the
// MMA warp and the consumers): as many as a group's kGC columns hold, at most 8. A group's tiles
// belong to one segment, hence to one expert slot, so they share the width.
struct GroupShape {
  int w, gt;
};
// B rows of tile t (its tokens' pieces, padded)
template <int NR>
__device__ __forceinline__ int tile_rows(const KParams& p, const WMisc* m, int kind, const WGeo& g, int t) {
  return min(NR, brows(tile_tokens(p, m, kind, g, t)));
}
// tiles of the slot that starts at tile t (< t1): two when both have at most pair_rows B rows
template <int NR>
__device__ __forceinline__ int slot_take(const KParams& p, const WMisc* m, int kind, const WGeo& g, int t, int t1) {
  return (t + 1 < t1 && tile_rows<NR>(p, m, kind, g, t) <= pair_rows(NR) &&
          tile_rows<NR>(p, m, kind, g, t + 1) <= pair_rows(NR)) ? 2 : 1;
}
// Slots of the tile range [t0, t1) under slot_take's rule: consecutive tiles of at most
// pair_rows rows pair up from the start of each run of them; a wider tile takes a slot alone.
// O(expert slots the range spans): an expert's tiles share their row count.
template <int NR>
__device__ int range_slots(const KParams& p, const WMisc* m, int kind, const WGeo& g, int t0, int t1) {
  if (t1 <= t0) return 0;
  if (kind != K_RTGU && kind != K_D) {
    const int n = t1 - t0;
    return tile_rows<NR>(p, m, kind, g, t0) <= pair_rows(NR) ? (n + 1) / 2 : n;
  }
  int slots = 0, run = 0;  // run: tiles of the current run of narrow tiles
  for (int u = t0 / g.tpe; u * g.tpe < t1; ++u) {
    const int a = max(t0, u * g.tpe), b = min(t1, (u + 1) * g.tpe);
    if (tile_rows<NR>(p, m, kind, g, a) <= pair_rows(NR)) {
      run += b - a;
    } else {
      slots += (run + 1) / 2 + (b - a);
      run = 0;
    }
  }
  return slots + (run + 1) / 2;
}

// byte offset of tile j's B block in a slot of n tiles
template <int NR>
__device__ __forceinline__ int b_off(int n, int j) { return n == 2 ? 2 * kTileBytes + j * (b_area(NR) / 2) : kTileBytes; }

// min(8, kGC / w) for B rows w = 16, 32, .., 128 (without a division)
static_assert(kGC == 256, "group_tiles assumes 256 columns per group");
__device__ __forceinline__ int group_tiles(int w) { return w <= 32 ? 8 : w == 48 ? 5 : w == 64 ? 4 : w == 80 ? 3 : 2; }
template <int NR>
__device__ __forceinline__ GroupShape group_shape(const KParams& p, const WMisc* m, int kind, const WGeo& g, int t) {
  GroupShape s;
  s.w = min(NR, brows(tile_tokens(p, m, kind, g, t)));
  s.gt = group_tiles(s.w);
  return s;
}

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
  static constexpr int PBS = NR * 128, SB = slot_bytes(NR);
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
  unsigned long long tw_fl = 0, tw_rel = 0;  // diagnostics: wait totals
  bool tw_on = false;
  __device__ bool claim(int& slot, bool mma_use) {
    const unsigned long long c0 = (DEC_TRACE && tw_on) ? gtimer() : 0;
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
    const unsigned long long c1 = (DEC_TRACE && tw_on) ? gtimer() : 0;
    if (plap > 0) {
      const bool pm = (last_mma & bit) != 0;
      const unsigned par = (((pm ? nm_par : ne_par) >> slot) & 1u) ^ 1u;
      if (!mbar_wait(pm ? &mempty[slot] : &empty[slot], par, p, 43)) {
        dead = true;
        return false;
      }
    }
    if (DEC_TRACE && tw_on) {
      tw_fl += c1 - c0;
      tw_rel += gtimer() - c1;
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
    if (kind == K_RTGU) return w.pbg + ((size_t)(t / g.tpe) * p.kb_d + kb) * PBS;
    return w.pbx + (size_t)kb * PBS;
  }

  __device__ void issue_gemv(int kind, int l, int U, const int* elist) {
    if (dead) return;
    WGeo g = wgeo(p, kind, U, gridDim.x);
    wsplit(g, m, p, kind, U, gridDim.x);
    const int t0 = wstart(g, blockIdx.x, gridDim.x), t1 = wstart(g, blockIdx.x + 1, gridDim.x);
    const LayerDev& Ld = p.layers[l < p.L ? l : 0];
    // Tile sources walked incrementally (the same as tile_src / b_src / slot_take give, without
    // a division or popcount per tile): the segment start (k block kb = t - seg0), the expert
    // slot u of tile t with its first tile, weights and B rows.
    const bool ex = kind == K_RTGU || kind == K_D;
    int seg0 = (t0 / g.kbs) * g.kbs;
    int u = ex ? t0 / g.tpe : 0;
    int u0 = ex ? u * g.tpe : 0, u1 = ex ? u0 + g.tpe : t1;
    auto rows_of = [&](int uu) { return min(NR, brows(ex ? __popcll(m->umask[uu]) : p.B)); };
    auto wbase = [&](int uu) -> const uint8_t* {
      switch (kind) {
        case K_QKV: return Ld.qkv;
        case K_O: return Ld.o;
        case K_ROUTER: return Ld.router;
        case K_SHGU: return Ld.sh_gu;
        case K_RTGU: return Ld.e_gu + (size_t)elist[uu] * p.e_gu_stride;
        case K_D: return uu < U ? Ld.e_d + (size_t)elist[uu] * p.e_d_stride : Ld.sh_d;
        default: return p.lm;
      }
    };
    auto bbase = [&](int uu) -> const uint8_t* {
      switch (kind) {
        case K_O: return w.pbo;
        case K_D: return w.pbh + (size_t)uu * p.kb_i * PBS;
        case K_RTGU: return w.pbg + (size_t)uu * p.kb_d * PBS;
        default: return w.pbx;
      }
    };
    int rows_u = t0 < t1 ? rows_of(u) : 0;
    const uint8_t* wb = t0 < t1 ? wbase(u) : nullptr;
    const uint8_t* bbs = t0 < t1 ? bbase(u) : nullptr;
    auto advance_to = [&](int t) {
      while (t >= seg0 + g.kbs) seg0 += g.kbs;
      while (t >= u1) {
        ++u;
        u0 = u1;
        u1 += g.tpe;
        rows_u = rows_of(u);
        wb = wbase(u);
        bbs = bbase(u);
      }
    };
    for (int t = t0; t < t1;) {
      int slot;
      if (!claim(slot, true)) return;
      advance_to(t);
      const int r1 = t + 1 < u1 ? rows_u : (t + 1 < t1 ? rows_of(u + 1) : 0);
      const int n = (t + 1 < t1 && rows_u <= pair_rows(NR) && r1 <= pair_rows(NR)) ? 2 : 1;  // (slot_take)
      const uint8_t* a[2];
      const uint8_t* b[2];
      unsigned bb[2];  // B bytes of each tile: its tokens' rows
      unsigned tx = 0;
      bool ok = true;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        if (j < n) {
          if (j) advance_to(t + 1);
          a[j] = wb + (size_t)(t + j - u0) * kTileBytes;
          b[j] = bbs + (size_t)(t + j - seg0) * PBS;
          bb[j] = (unsigned)rows_u * 128u;
          tx += kTileBytes + bb[j];
          ok = ok && within(a[j], kTileBytes, p.warena, p.warena_bytes) && within(b[j], bb[j], w.pb, w.pb_bytes);
        }
      }
      t += n;
      uint8_t* dst = ring + (size_t)slot * SB;
      if (!ok) {
        raise_err(p, kDevBadArg, 45);
        mbar_arrive(&full[slot]);
        advance();
        continue;
      }
      mbar_arrive_expect_tx(&full[slot], tx);
      if (n == 2 && a[1] == a[0] + kTileBytes) {
        bulk_g2s_hint(dst, a[0], 2 * kTileBytes, &full[slot], pol_stream);
      } else {
        for (int j = 0; j < n; ++j) bulk_g2s_hint(dst + (size_t)j * kTileBytes, a[j], kTileBytes, &full[slot], pol_stream);
      }
      for (int j = 0; j < n; ++j) bulk_g2s_hint(dst + b_off<NR>(n, j), b[j], bb[j], &full[slot], pol_near);
      advance();
    }
  }

  // KV tiles of the CTA's attention units (rows before the new position: written by earlier
  // launches; the unit patches the new position into its copy)
  __device__ void issue_attn(int l) {
    if (dead) return;
    const int NU = p.B * p.hkv * w.nch;
    const int planes = p.L * p.slots * p.hkv;
    for (int u = blockIdx.x; u < NU; u += gridDim.x) {
      const WUnit a = wunit(p, w, m, u);
      const int z = (l * p.slots + p.seq0 + a.b) * p.hkv + a.g;  // (the rows of kv_row)
      for (int t = a.tile0; t < a.tile1; t += 2) {  // a round: its K, then its V
        const int p0 = t * kKvTilePos;
#pragma unroll 1
        for (int kv = 0; kv < 2; ++kv) {
          int slot;
          if (!claim(slot, false)) return;
          uint8_t* dst = kv_area(ring + (size_t)slot * SB);
          if (a.T - p0 < 1 || a.T > p.max_ctx || z < 0 || z >= planes) {
            raise_err(p, kDevBadArg, 46);
            mbar_arrive(&full[slot]);
            advance();
            continue;
          }
          // whole boxes of both tiles (rows past the cache's end read as zeros)
          mbar_arrive_expect_tx(&full[slot], 2u * kKvTilePos * HD * 2);
#pragma unroll
          for (int hb = 0; hb < HD / 64; ++hb)
#pragma unroll
            for (int i = 0; i < 2; ++i)
              tma_load_3d(dst + hb * 16384 + i * 8192, kv ? &w.vmap : &w.kmap, hb * 64, p0 + i * kKvTilePos, z,
                          &full[slot], pol_near);
          advance();
        }
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
        if (!wait_bar(base + 8)) break;  // (the slots' tokens gathered)
        tw_on = true;
        issue_gemv(K_RTGU, l, U, elist);
        tw_on = false;
      }
      if (!wait_bar(base + 10)) break;
      issue_gemv(K_D, l, U, elist);
      ++lay;
    }
    if (p.V > 0 && !dead && wait_bar(1u + (unsigned)(kBarsPerLayer * p.L))) issue_gemv(K_LM, 0, 0, elist);
    drain();
    if (DEC_TRACE && blockIdx.x == 0) {
      p.trace[kWaitTrace + 0] = tw_fl;
      p.trace[kWaitTrace + 1] = tw_rel;
    }
  }
};

// ---------------------------------------------------------------------------------------------
// MMA warp (one thread): the CTA's tiles in the consumers' order, in groups of tiles of one
// segment (group_shape: as many as kGC TMEM columns hold), kNGW groups in flight.

template <int NR, int HD, int G>
struct WMma {
  static constexpr int SB = slot_bytes(NR);
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
  unsigned long long tw_full = 0, tw_tmem = 0;  // diagnostics: wait totals in routed gate/up stages
  // diagnostics: its stage time, MMA issue time and tiles in the routed gate/up and down stages
  unsigned long long tw_mstage[2] = {0, 0}, tw_miss[2] = {0, 0}, tw_mtiles[2] = {0, 0};
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
    const int dk = kind == K_D ? 1 : 0;
    const bool twx = DEC_TRACE && (kind == K_RTGU || kind == K_D);
    const unsigned long long cs = twx ? gtimer() : 0;
    WGeo g = wgeo(p, kind, U, gridDim.x);
    wsplit(g, m, p, kind, U, gridDim.x);
    const int t0 = wstart(g, blockIdx.x, gridDim.x), t1 = wstart(g, blockIdx.x + 1, gridDim.x);
    int j = 0, ns = 0;  // tile j of the current slot of ns tiles
    // The same tile, slot and group sequence as slot_take / group_shape give, walked
    // incrementally (this warp's bookkeeping paces the expert stages at large batches: integer
    // divisions and popcounts per tile cost more than the tile's MMAs): the segment's end, the
    // expert slot's end and its B rows follow t.
    const bool ex = kind == K_RTGU || kind == K_D;
    int seg_end = (t0 / g.kbs + 1) * g.kbs;
    int u = ex ? t0 / g.tpe : 0;
    int u_end = ex ? (u + 1) * g.tpe : t1;
    auto rows_of = [&](int uu) { return min(NR, brows(ex ? __popcll(m->umask[uu]) : p.B)); };
    int rows_u = t0 < t1 ? rows_of(u) : 0;
#pragma unroll 1
    for (int t = t0; t < t1;) {
      while (t >= seg_end) seg_end += g.kbs;
      while (t >= u_end) {
        ++u;
        u_end += g.tpe;
        rows_u = rows_of(u);
      }
      const GroupShape gs{rows_u, group_tiles(rows_u)};
      const int n = min(gs.gt, min(t1, seg_end) - t);
      const int gsl = gseq % kNGW;
      const bool tw = DEC_TRACE && kind == K_RTGU;
      unsigned long long c0 = tw ? gtimer() : 0;
      if (!dead && gseq >= (unsigned)kNGW && !mbar_wait(&m->tempty[gsl], (gseq / kNGW - 1) & 1, p, 48)) dead = true;
      if (tw) tw_tmem += gtimer() - c0;
#pragma unroll 1
      for (int i = 0; i < n; ++i, ++t) {
        if (j == 0) {  // (slot_take)
          const int r1 = t + 1 < u_end ? rows_u : (t + 1 < t1 ? rows_of(u + 1) : 0);
          ns = (t + 1 < t1 && rows_u <= pair_rows(NR) && r1 <= pair_rows(NR)) ? 2 : 1;
          if (tw) c0 = gtimer();
          if (!dead && !mbar_wait(&full[slot], lap & 1, p, 49)) dead = true;
          if (tw) tw_full += gtimer() - c0;
        }
        const uint8_t* a = ring + (size_t)slot * SB + (size_t)j * kTileBytes;
        const uint8_t* b = ring + (size_t)slot * SB + b_off<NR>(ns, j);
        const unsigned long long ci = twx ? gtimer() : 0;
        if (!dead) {
          tc_fence_after();
          m->hdr[gsl][i] = *reinterpret_cast<const float2*>(a + kTileData);
          const uint64_t ad = smem_desc(a, 128, 1024), bd = smem_desc(b, 128, 1024);
          const uint32_t d = tmem + (uint32_t)(gsl * kGC + i * gs.w);
          const uint32_t idesc = idesc_e4m3_f32(kTileRows, gs.w);
#pragma unroll
          for (int k = 0; k < kTileK / 32; ++k)
            mma_e4m3(d, ad + (uint64_t)(k * 16), bd + (uint64_t)(k * 16), idesc, k > 0 ? 1u : 0u);
        }
        if (twx) {
          tw_miss[dk] += gtimer() - ci;
          ++tw_mtiles[dk];
        }
        if (++j == ns) {
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
    if (twx) tw_mstage[dk] += gtimer() - cs;
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
        items += 2 * ((a.tile1 - a.tile0 + 1) / 2);  // (a K and a V item per round of two tiles)
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
    if (DEC_TRACE && blockIdx.x == 0) {
      p.trace[kWaitTrace + 2] = tw_full;
      p.trace[kWaitTrace + 3] = tw_tmem;
      for (int i = 0; i < 2; ++i) {
        p.trace[kWaitTrace + 20 + 3 * i] = tw_mstage[i];
        p.trace[kWaitTrace + 21 + 3 * i] = tw_miss[i];
        p.trace[kWaitTrace + 22 + 3 * i] = tw_mtiles[i];
      }
    }
    mbar_arrive(&m->mma_done);
  }
};

// ---------------------------------------------------------------------------------------------
// consumer warps

template <int NR, int HD, int G>
struct WConsumer {
  static constexpr int PBS = NR * 128, SB = slot_bytes(NR);
  static constexpr int TPT = NR / 4;  // tokens per thread in a tile's epilogue
  float4* acc4 = nullptr;  // the GEMV accumulators [token chunk][warp half][row] (shared memory)
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
  unsigned long long tw_prod = 0, tw_stage = 0, tw_ld = 0, tw_flush = 0;  // diagnostics (thread 0): routed gate/up
  unsigned long long tw_dprod = 0, tw_dstage = 0, tw_dflush = 0;  // the same in the down projection
  int rtgu_seen = 0;
  unsigned sph = 0, oph = 0;  // attention MMA completions waited for (phases of sbar, obar)
  unsigned long long tw_kv = 0, tw_attn = 0, tw_pro = 0, tw_post = 0;  // diagnostics: attention
  unsigned long long tw_a[8] = {0, 0, 0, 0, 0, 0, 0, 0};  // diagnostics: attention round steps
  uint32_t tmem = 0;

  __device__ WConsumer(const KParams& p_, const WideParams& w_, uint8_t* r, uint64_t* f, uint64_t* e, float* rd,
                       WMisc* m_, float4* a4)
      : p(p_), w(w_), ring(r), full(f), empty(e), red(rd), m(m_), acc4(a4) {
    tid = threadIdx.x;
    warp = tid >> 5;
    lane = tid & 31;
  }

  __device__ const uint8_t* wait_item() {
    const unsigned long long c0 = DEC_TRACE ? gtimer() : 0;
    if (!dead && !mbar_wait(&full[rslot], rpar, p, 52)) dead = true;
    if (DEC_TRACE && tid == 0) tw_kv += gtimer() - c0;
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
    // (tests only: CTA 0 withholds its arrival at the first barrier, so every wait runs out)
    const bool withhold = p.test_skip && nbar == 1 && blockIdx.x == 0;
    if (tid == kPubThread && !dead && !withhold) red_release_add(reinterpret_cast<int*>(w.bar), 1);
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
    // diagnostics build: CTA 0's time at each grid barrier (phase boundaries)
    if (DEC_TRACE && blockIdx.x == 0 && tid == 0 && nbar < (unsigned)kTraceSlots) p.trace[nbar] = gtimer();
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

  // Add the products of group gs (n consecutive tiles of one segment, from tile t: one expert
  // slot, k blocks kb0 .. kb0 + n - 1) into the thread's accumulators. The tile's tokens (the
  // step's, or the expert slot's in ascending order) come in chunks of 8 (16 TMEM columns, token
  // j's pieces in columns 2j, 2j + 1); the two warps of a TMEM lane quadrant (w, w + 4) take 4
  // tokens of each chunk: thread (warp w, lane) holds weight row 32 (w & 3) + lane of tokens
  // 8c + 4 (w >> 2) + j, accumulator 4c + j. The loads of two tiles are issued before one wait.
  // Each product is scaled by the tile's block scale and the pieces' 2^-a.
  static constexpr int LB = 2;
  __device__ __forceinline__ void epilogue(unsigned gs, int n, int sw, int kind, const WGeo& g, int t, int u_lo,
                                          int) {
    const int gsl = gs % kNGW;
    const unsigned long long c0 = (DEC_TRACE && (kind == K_RTGU || kind == K_D)) ? gtimer() : 0;
    if (!dead && !mbar_wait(&m->tfull[gsl], (gs / kNGW) & 1, p, 54)) dead = true;
    if (DEC_TRACE && kind == K_RTGU && tid == 0) tw_prod += gtimer() - c0;
    if (DEC_TRACE && kind == K_D && tid == 0) tw_dprod += gtimer() - c0;
    dead = __any_sync(0xffffffffu, dead);  // (the TMEM loads below are warp-collective)
    const int q = warp & 3, h = warp >> 2, row = 32 * q + lane;
    const int seg = t / g.kbs, kb0 = t - seg * g.kbs;
    const int ntok = tile_tokens(p, m, kind, g, t);  // (the group's tiles share it)
    const int xr0 = (kind == K_RTGU || kind == K_D) ? (t / g.tpe - u_lo) * g.kbs + kb0 : kb0;
    if (!dead) {
      tc_fence_after();
      const uint32_t tb = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(gsl * kGC + 8 * h);
#pragma unroll
      for (int c = 0; c < NR / 16; ++c) {
        if (8 * c + 4 * h >= ntok) break;  // (warp-uniform)
        float a4[4] = {0.f, 0.f, 0.f, 0.f};  // the group's sum for this chunk
#pragma unroll 1
        for (int i0 = 0; i0 < n; i0 += LB) {
          const int nb = min(LB, n - i0);
          uint32_t d[LB][8];
          const uint32_t ta = tb + (uint32_t)(i0 * sw + 16 * c);
          const unsigned long long cl = (DEC_TRACE && kind == K_RTGU) ? gtimer() : 0;
          if (nb == 2) tmem_ld8x2_wait(ta, ta + (uint32_t)sw, d);
          else tmem_ld8_wait(ta, d[0]);
          if (DEC_TRACE && kind == K_RTGU && tid == 0) tw_ld += gtimer() - cl;
#pragma unroll
          for (int k = 0; k < LB; ++k) {
            if (k < nb) {
              const int i = i0 + k;
              const float2 sc = m->hdr[gsl][i];
              const float s_r = row < 64 ? sc.x : sc.y;
              const uint32_t e4 = *reinterpret_cast<const uint32_t*>(m->ex + (xr0 + i) * kWideMax + 8 * c + 4 * h);
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const int a = (int)(int8_t)(e4 >> (8 * j));
                const float inv = __int_as_float((127 - a) << 23);
                const float v = fmaf(__uint_as_float(d[k][2 * j + 1]), 0.0625f, __uint_as_float(d[k][2 * j]));
                a4[j] = fmaf(s_r * inv, v, a4[j]);
              }
            }
          }
        }
        float4& dst = acc4[(c * 2 + h) * kTileRows + row];
        dst = make_float4(dst.x + a4[0], dst.y + a4[1], dst.z + a4[2], dst.w + a4[3]);
      }
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&m->tempty[gsl]);
  }

  // token t's gate for expert slot u: its selections' slots as one 8-byte word, the matching
  // byte found without a loop (a token selects a slot at most once)
  __device__ float gate_of(int t, int u) const {
    static_assert(kWideTopk == 8, "one 8-byte word of selections per token");
    const unsigned long long x =
        *reinterpret_cast<const unsigned long long*>(m->wsel[t]) ^ (0x0101010101010101ull * (unsigned)u);
    const unsigned long long z = (x - 0x0101010101010101ull) & ~x & 0x8080808080808080ull;  // zero bytes
    if (z == 0ull) return 0.f;
    const int k = (__ffsll((long long)z) - 1) >> 3;  // (the lowest zero byte is found exactly)
    return k < p.topk ? m->wgate[t][k] : 0.f;
  }

  // One segment's partial sums of the CTA: plain stores (read after the next grid barrier), per
  // token of the step. Routed stages: the expert slot's j-th token is tl[u][j]; the down
  // projection's partials carry that token's gate.
  __device__ __forceinline__ void flush(int kind, const WGeo& g, int seg, int first, int U) {
    if (dead) return;
    const int slot = wcontrib_slot(g, blockIdx.x, first, seg, gridDim.x);
    float* dst = part_of(p, kind) + (size_t)(seg * g.S + slot) * p.MB * kTileRows;
    const int row = 32 * (warp & 3) + lane, h = warp >> 2;
    // accumulator 4c + j holds the tile's token 8c + 4h + j
    if (kind == K_RTGU || kind == K_D) {
      const int u = seg / (kind == K_RTGU ? p.n_rb_gu : p.n_rb_d);
      const int n = __popcll(m->umask[u]);
      const uint8_t* tl = slot_tokens() + u * kWideMax + 4 * h;
#pragma unroll
      for (int k = 0; k < TPT; ++k) {
        const int jl = 8 * (k >> 2) + (k & 3);  // (local token 8c + 4h + j, minus 4h)
        if (jl + 4 * h < n) {
          const int t = tl[jl];
          float v = acc_get(k, h, row);
          if (kind == K_D && u < U) v *= gate_of(t, u);
          dst[(size_t)t * kTileRows + row] = v;
        }
      }
      return;
    }
    // (the thread's tokens: one base address, constant offsets)
    float* base = dst + (size_t)4 * h * kTileRows + row;
    const int nb = p.B - 4 * h;
#pragma unroll
    for (int k = 0; k < TPT; ++k) {
      const int jl = 8 * (k >> 2) + (k & 3);
      if (jl < nb) base[jl * kTileRows] = acc_get(k, h, row);
    }
  }

  // accumulator k (token 8 (k / 4) + 4 h + k % 4) of the thread (row, half h)
  __device__ __forceinline__ float acc_get(int k, int h, int row) const {
    const float4 a = acc4[((k >> 2) * 2 + h) * kTileRows + row];
    return (k & 3) == 0 ? a.x : (k & 3) == 1 ? a.y : (k & 3) == 2 ? a.z : a.w;
  }

  // shared-memory tables of the routing phases (in red): expert marks, the SwiGLU (slot, token)
  // pairs, each slot's tokens in ascending order
  __device__ __forceinline__ int* route_marks() const { return reinterpret_cast<int*>(red); }
  __device__ __forceinline__ int* swiglu_pairs() const { return reinterpret_cast<int*>(red) + kMaxExperts; }
  __device__ __forceinline__ uint8_t* slot_tokens() const {
    return reinterpret_cast<uint8_t*>(reinterpret_cast<int*>(red) + kMaxExperts + kWideMax * 17);
  }

  __device__ void gemv(int kind, int U) {
    const unsigned long long cs = (DEC_TRACE && (kind == K_RTGU || kind == K_D)) ? gtimer() : 0;
    WGeo g = wgeo(p, kind, U, gridDim.x);
    wsplit(g, m, p, kind, U, gridDim.x);
    const int t0 = wstart(g, blockIdx.x, gridDim.x), t1 = wstart(g, blockIdx.x + 1, gridDim.x);
    // the exponents of the B blocks the CTA's tiles read (written before the last barrier)
    int u_lo = 0;
    if (t1 > t0 && !dead) {
      const int8_t* src;
      int rows;
      if (kind == K_D || kind == K_RTGU) {
        u_lo = t0 / g.tpe;
        const int u_hi = (t1 - 1) / g.tpe;
        rows = (u_hi - u_lo + 1) * g.kbs;
        src = (kind == K_D ? w.exh : w.exg) + (size_t)u_lo * g.kbs * kWideMax;
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
    int seg_cur = -1, seg_first = 0;
#pragma unroll 1
    for (int t = t0;;) {
      const int seg = t < t1 ? t / g.kbs : -1;
      if (t == t1 || seg != seg_cur) {
        const unsigned long long cf = (DEC_TRACE && (kind == K_RTGU || kind == K_D)) ? gtimer() : 0;
        if (seg_cur >= 0) flush(kind, g, seg_cur, seg_first, U);
        if (DEC_TRACE && kind == K_RTGU && tid == 0) tw_flush += gtimer() - cf;
        if (DEC_TRACE && kind == K_D && tid == 0) tw_dflush += gtimer() - cf;
        if (t == t1) break;
        seg_cur = seg;
        seg_first = t;
        {
          const int row = 32 * (warp & 3) + lane, h = warp >> 2;
#pragma unroll
          for (int c = 0; c < NR / 16; ++c) acc4[(c * 2 + h) * kTileRows + row] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
      const GroupShape gsh = group_shape<NR>(p, m, kind, g, t);
      const int n = min(gsh.gt, min(t1, (seg + 1) * g.kbs) - t);
      epilogue(gseq++, n, gsh.w, kind, g, t, u_lo, 0);
      t += n;
    }
    // the stage's slots (freed by the MMA warp): keep the ring position in step
    ring_skip(range_slots<NR>(p, m, kind, g, t0, t1));
    dead = cons_any(dead);
    if (DEC_TRACE && kind == K_D && tid == 0) tw_dstage += gtimer() - cs;
    if (DEC_TRACE && kind == K_RTGU && tid == 0) {
      const unsigned long long dt = gtimer() - cs;
      tw_stage += dt;
      if (DEC_STAMPS && ++rtgu_seen == 4) {  // (layer 3: start and end of every CTA's stage)
        p.trace[kTraceSlots + blockIdx.x] = cs;
        p.trace[kTraceSlots + gridDim.x + blockIdx.x] = cs + dt;
      }
    }
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

  // eight bf16 values (given as floats that bf16 holds exactly) as one 16-byte chunk
  __device__ __forceinline__ static uint4 bf16x8(const float* f) {
    uint32_t u[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) u[i] = (uint32_t)f2bf(f[2 * i]) | ((uint32_t)f2bf(f[2 * i + 1]) << 16);
    return make_uint4(u[0], u[1], u[2], u[3]);
  }

  // Split-context GQA decode on the tensor cores: unit (token b, KV head g, chunk c) over the KV
  // tiles of its chunk in rounds of two 64-position tiles, one online softmax per unit. For a
  // round the producer loads K into one ring slot and V into the next with tensor-map copies, in
  // the 128-byte swizzled layout the MMAs read (128 positions of both tiles in a row); the
  // consumers only write in the new position's key and value (and zero the value rows past it).
  // One thread issues S^T = K q^T (M = the round's 128 positions, N = 16 columns: the group's
  // heads, then zeros; bf16 operands, fp32 in TMEM columns 0..15). Each thread takes its
  // position's scores, each head's maximum over the round, forms p = 2^(s - m) and splits it into
  // three bf16 pieces, p = p1 + p2 + p3 within 2^-27 p (two pieces, within 2^-17 p, flipped the
  // bf16 rounding of about one output in a thousand against fp32 arithmetic); one thread issues
  // O^T = V^T [p1 p2 p3] (M = head_dim rows, V read MN-major; TMEM columns 16..31) and each
  // output row's thread rescales its running sum and adds the pieces' products. An MMA of these
  // shapes costs tens of nanoseconds whatever its N, so a round takes 2 x head_dim / 16 of them
  // for 128 positions. One chunk: the normalised outputs go straight to the B blocks of the
  // projection; otherwise the chunk's state is published for the merge phase.
  static constexpr int NCH = HD / 8;           // 16-byte chunks of a K or V row
  static constexpr int NT = kConsumerWarps * 32;

  // the ring item after the current one (the current one still held)
  __device__ const uint8_t* wait_next_item() {
    int s = rslot + 1;
    unsigned par = rpar;
    if (s == p.ring) {
      s = 0;
      par ^= 1;
    }
    if (!dead && !mbar_wait(&full[s], par, p, 52)) dead = true;
    return ring + (size_t)s * SB;
  }

  __device__ __forceinline__ static float warp_max(float v) {
    float r;
    asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
    return r;
  }

  // O^T of the round just finished (TMEM columns 16..): this output row's running sums rescaled
  // by the round's factors, then the three pieces' products added
  __device__ __forceinline__ void add_o(float (&acc)[G / 2], int h0) {
    const uint32_t ta = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + 16u;
    float o[16];
    if constexpr (3 * G > 8) {
      tmem_ld16(ta, o);
    } else {
      float o8[8];
      tmem_ld<8>(ta, o8);
#pragma unroll
      for (int i = 0; i < 16; ++i) o[i] = i < 8 ? o8[i] : 0.f;
    }
#pragma unroll
    for (int j = 0; j < G / 2; ++j) {
      const int h = h0 + j;
      acc[j] = acc[j] * m->acr[h] + (o[h] + (o[G + h] + o[2 * G + h]));
    }
  }

  __device__ void attention(int l) {
    static_assert(HD == 64 || HD == 128, "head_dim 64 or 128");
    static_assert(G % 2 == 0 && 3 * G <= 16, "two head groups; the three p pieces within 16 columns");
    constexpr int GH = G / 2;                     // heads per warp group
    constexpr int HB = HD / 64;                   // 64-wide d parts of a round's K or V
    uint8_t* st = reinterpret_cast<uint8_t*>(acc4);
    uint8_t* ps = st + att_p(HD);
    uint8_t* qs = st + att_q(HD);
    const float qscale = 1.4426950408889634f / sqrtf((float)HD);
    const int NU = p.B * p.hkv * w.nch;
    const int q4 = warp & 3, h0 = (warp >> 2) * GH;  // TMEM lane quadrant; the warp's heads
    const bool out_warp = 32 * q4 < HD;  // TMEM lanes 0..HD-1: output rows d
    const uint32_t tl = tmem + ((uint32_t)(32 * q4) << 16);
    constexpr uint32_t kIdS = idesc_bf16_f32(128, 16, false), kIdO = idesc_bf16_f32(128, 16, true);
    // S^T = K q^T. A = K, K-major 128-byte swizzled (8-row groups 1024 B apart; K = 16 steps of 32
    // bytes inside a 64-wide d part, then the next part); B = q ([d chunk][row][8 values]: rows 8 apart 128 B,
    // d chunks 256 B).
    auto issue_s = [&](const uint8_t* kk) {
      const uint64_t bd = smem_desc(qs, 256, 128);
#pragma unroll
      for (int k = 0; k < HD / 16; ++k)
        mma_bf16(tmem, smem_desc_sw128(kk + (k >> 2) * 16384 + (k & 3) * 32, 16, 1024), bd + (uint64_t)(k * 32), kIdS,
                 k > 0 ? 1u : 0u);
    };
    // O^T = V^T P. A = V^T, MN-major 128-byte swizzled (64-row atoms of d one part apart, groups
    // of 8 positions 1024 B); B = P ([position block][column][8 positions]: columns 8 apart 128 B,
    // position blocks 256 B).
    auto issue_o = [&](const uint8_t* vv) {
      const uint64_t bd = smem_desc(ps, 256, 128);
#pragma unroll
      for (int k = 0; k < 2 * kKvTilePos / 16; ++k)
        mma_bf16(tmem + 16, smem_desc_sw128(vv + k * 2048, 16384, 1024), bd + (uint64_t)(k * 32), kIdO,
                 k > 0 ? 1u : 0u);
    };
    const unsigned long long ca = DEC_TRACE ? gtimer() : 0;
#pragma unroll 1
    for (int u = blockIdx.x; u < NU; u += gridDim.x) {
      const WUnit a = wunit(p, w, m, u);
      float* qkvn = red;
      const unsigned long long cp = DEC_TRACE ? gtimer() : 0;
      if (a.tile1 > a.tile0) prologue(l, a, qkvn);  // (CTA barriers inside: no branch on `dead`)
      if (DEC_TRACE && tid == 0) tw_pro += gtimer() - cp;
      // the group's query heads in rows 0..G-1 of q's staging, zero rows after; P zeroed
      for (int i = tid; i < NCH * 16; i += NT) {
        const int dc = i >> 4, n = i & 15;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (n < G && a.tile1 > a.tile0) v = bf16x8(qkvn + n * HD + dc * 8);
        *reinterpret_cast<uint4*>(qs + dc * 256 + n * 16) = v;
      }
      for (int i = tid; i < kKvTilePos * 4; i += NT) reinterpret_cast<uint4*>(ps)[i] = make_uint4(0u, 0u, 0u, 0u);
      float acc[GH], mrun[GH], lw[GH];  // lw: this lane's position's share of the sums
#pragma unroll
      for (int j = 0; j < GH; ++j) {
        acc[j] = 0.f;
        mrun[j] = -INFINITY;
        lw[j] = 0.f;
      }
      const int newpos = a.T - 1;
      // The tile that holds the new position: its key and value rows written in (the cache copy
      // may predate the prologue's append), value rows after it zeroed (the cache there may hold
      // anything; P is 0 there, but 0 x NaN would not be). After the tile has landed.
      auto patch = [&](uint8_t* kk, uint8_t* vv, int jn) {  // (jn: the row in the round, < 128)
        const int nk = HB * 8, nv = (2 * kKvTilePos - jn) * HB * 8;
        for (int i = tid; i < nk + nv; i += NT) {
          const bool isk = i < nk;
          const int ii = isk ? i : i - nk;
          const int c = ii & 7, hb = (ii >> 3) % HB, r = isk ? jn : jn + (ii >> 3) / HB;
          uint4 v = make_uint4(0u, 0u, 0u, 0u);
          if (isk) v = bf16x8(qkvn + G * HD + hb * 64 + c * 8);
          else if (r == jn) v = bf16x8(qkvn + (G + 1) * HD + hb * 64 + c * 8);
          *reinterpret_cast<uint4*>((isk ? kk : vv) + hb * 16384 + r * 128 + ((c ^ (r & 7)) << 4)) = v;
        }
      };
      // rounds of two tiles (the second may lie past the chunk or the context: masked): S^T of
      // both in one M = 128 product, one softmax over their 128 positions, O^T over both
      const int pend = min(a.T, a.tile1 * kKvTilePos);  // this unit's positions end here
#pragma unroll 1
      for (int t = a.tile0; t < a.tile1; t += 2) {
        unsigned long long c0 = DEC_TRACE ? gtimer() : 0, c1 = 0;
#define ATT_T(i) if (DEC_TRACE && tid == 0) { c1 = gtimer(); tw_a[i] += c1 - c0; c0 = c1; }
        uint8_t* kk = kv_area(const_cast<uint8_t*>(wait_item()));
        uint8_t* vv = kv_area(const_cast<uint8_t*>(wait_next_item()));
        const int p0 = t * kKvTilePos;
        const int jn = newpos - p0;  // (the new position is in this round if jn < 128)
        const bool patched = jn < 2 * kKvTilePos;
        if (patched && !dead) patch(kk, vv, jn);
        if (patched || t == a.tile0) fence_proxy_async_smem();  // (the first round: q and P staging too)
        ATT_T(0)
        tc_fence_before();
        cons_sync();
        if (tid == 0) {
          tc_fence_after();
          if (!dead) issue_s(kk);
          mma_commit(&m->sbar);
        }
        ATT_T(1)
        if (!dead && !mbar_wait(&m->sbar, sph & 1u, p, 57)) dead = true;
        ATT_T(2)
        ++sph;
        tc_fence_after();
        release_item();  // (the K slot: its product is done; the producer may refill it now)
        // scores: this lane's position (TMEM lane) of the round; each head's maximum
        const int pos = 32 * q4 + lane;
        float sv[GH];
        {
          float s8[8];
          tmem_ld<G>(tl, s8);
#pragma unroll
          for (int j = 0; j < GH; ++j) {
            sv[j] = p0 + pos < pend ? s8[h0 + j] * qscale : -INFINITY;
            const float mx = warp_max(sv[j]);
            if (lane == 0) m->amx[q4][h0 + j] = mx;
          }
        }
        tc_fence_before();
        cons_sync();
        ATT_T(3)
        // softmax of the round: P's three pieces, the rescale factors
        {
          uint8_t* pr = ps + (pos >> 3) * 256 + (pos & 7) * 2;  // [position block][column][8 positions]
#pragma unroll
          for (int j = 0; j < GH; ++j) {
            const int h = h0 + j;
            const float mr = fmaxf(fmaxf(m->amx[0][h], m->amx[1][h]), fmaxf(m->amx[2][h], m->amx[3][h]));
            const float mnew = fmaxf(mrun[j], mr);
            const float corr = mrun[j] == -INFINITY ? 0.f : exp2f(mrun[j] - mnew);
            const float pe = sv[j] == -INFINITY ? 0.f : exp2f(sv[j] - mnew);
            const uint16_t p1 = f2bf(pe);
            const float r1 = pe - bf16f(p1);  // (exact, and r1 - bf16(r1) too)
            const uint16_t p2 = f2bf(r1);
            *reinterpret_cast<uint16_t*>(pr + h * 16) = p1;
            *reinterpret_cast<uint16_t*>(pr + (G + h) * 16) = p2;
            *reinterpret_cast<uint16_t*>(pr + (2 * G + h) * 16) = f2bf(r1 - bf16f(p2));
            lw[j] = lw[j] * corr + pe;
            mrun[j] = mnew;
            if (q4 == 0 && lane == 0) m->acr[h] = corr;
          }
          fence_proxy_async_smem();
        }
        cons_sync();
        ATT_T(4)
        if (tid == 0) {
          tc_fence_after();
          if (!dead) issue_o(vv);
          mma_commit(&m->obar);
        }
        ATT_T(5)
        if (!dead && !mbar_wait(&m->obar, oph & 1u, p, 58)) dead = true;
        ATT_T(6)
        ++oph;
        tc_fence_after();
        if (out_warp) add_o(acc, h0);
        tc_fence_before();
        release_item();  // (the V slot)
        ATT_T(7)
#undef ATT_T
      }
      // the unit's state per head: m (the same in every warp of a head group), l = the sum over
      // lanes and lane quadrants
#pragma unroll
      for (int j = 0; j < GH; ++j) {
        float s = lw[j];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
        if (lane == 0) {
          m->alw[q4][h0 + j] = s;
          if (q4 == 0) m->amr[h0 + j] = mrun[j];
        }
      }
      dead = cons_any(dead);  // (one verdict: the packing below is warp-collective)
      const unsigned long long cq = DEC_TRACE ? gtimer() : 0;
      if (w.nch == 1) {
        // the normalised output (bf16) of the group's heads, then their B blocks
        float* ob = red;
        if (out_warp) {
          const int d = 32 * q4 + lane;
#pragma unroll
          for (int j = 0; j < GH; ++j) {
            const int h = h0 + j;
            const float L = (m->alw[0][h] + m->alw[1][h]) + (m->alw[2][h] + m->alw[3][h]);
            const float wgt = (m->amr[h] == -INFINITY || !(L > 0.f)) ? 0.f : 1.f / L;
            ob[h * HD + d] = bf16f(f2bf(wgt * acc[j]));
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
      } else if (!dead && out_warp) {
        float* dst = w.attn_part + ((((size_t)a.b * p.hkv + a.g) * w.nch + a.c) * G) * (HD + 2);
        const int d = 32 * q4 + lane;
#pragma unroll
        for (int j = 0; j < GH; ++j) {
          const int h = h0 + j;
          dst[(size_t)h * (HD + 2) + d] = acc[j];
          if (d == 0) {
            dst[(size_t)h * (HD + 2) + HD] = m->amr[h];
            dst[(size_t)h * (HD + 2) + HD + 1] = (m->alw[0][h] + m->alw[1][h]) + (m->alw[2][h] + m->alw[3][h]);
          }
        }
      }
      cons_sync();
      if (DEC_TRACE && tid == 0) tw_post += gtimer() - cq;
    }
    if (DEC_TRACE && tid == 0) tw_attn += gtimer() - ca;
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
    int* mark = route_marks();
    int* pairs = swiglu_pairs();
    uint8_t* tl = slot_tokens();
    const unsigned long long all = p.B >= 64 ? ~0ull : ((1ull << p.B) - 1ull);
    if (p.dense) {
      if (tid == 0) {
        m->U = 0;
        m->umask[0] = all;
        m->npairs = p.B;
      }
      for (int t = tid; t < p.B; t += kConsumerWarps * 32) {
        pairs[t] = t;
        tl[t] = (uint8_t)t;
      }
      cons_sync();
      slot_weights(0);
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
    // each slot's tokens in ascending order (thread u scans its mask)
    for (int u = tid; u <= U; u += kConsumerWarps * 32) {
      unsigned long long mk = (u < U || p.nsh) ? m->umask[u] : 0ull;
      for (int j = 0; mk; ++j, mk &= mk - 1) tl[u * kWideMax + j] = (uint8_t)(__ffsll((long long)mk) - 1);
    }
    cons_sync();
    slot_weights(U);
    if (tid == 0) mbar_arrive(&m->rt_bar);  // the producer and the MMA warp may take the routed experts
  }

  // the expert slots' tile weights for the work-weighted split (wsplit): B rows / 16, at least 2
  __device__ void slot_weights(int U) {
    if (tid == 0) {
      int acc = 0, wm = 0;
      m->pw[0] = 0;
      for (int u = 0; u < U + p.nsh; ++u) {
        const int wu = max(2, min(NR, brows(__popcll(m->umask[u]))) / 16);
        acc += wu;
        m->pw[u + 1] = acc;
        wm = max(wm, wu);
      }
      m->wmax = wm;
    }
    cons_sync();
  }

  // The B rows of each routed slot's tokens, gathered from pbx into compact blocks (pbg, exg):
  // warp unit (slot u, k block kb) copies 2 x 8 16-byte chunks per token.
  __device__ void gather(int U) {
    const uint8_t* tl = slot_tokens();
    const int nw = gridDim.x * kConsumerWarps;
#pragma unroll 1
    for (int wu = blockIdx.x * kConsumerWarps + warp; wu < U * p.kb_d && !dead; wu += nw) {
      const int u = wu / p.kb_d, kb = wu % p.kb_d;
      const int n = __popcll(m->umask[u]);
      const uint8_t* src = w.pbx + (size_t)kb * PBS;
      uint8_t* dst = w.pbg + ((size_t)u * p.kb_d + kb) * PBS;
      for (int i = lane; i < 16 * n; i += 32) {
        const int r = i >> 3, c = (i & 7) * 16;  // local row r (token r / 2, piece r % 2), chunk c
        const int t = tl[u * kWideMax + (r >> 1)];
        *reinterpret_cast<uint4*>(dst + boff(r, c)) = ldcg4(src + boff(2 * t + (r & 1), c));
      }
      for (int j = lane; j < n; j += 32)
        w.exg[((size_t)u * p.kb_d + kb) * kWideMax + j] = __ldcg(w.exx + (size_t)kb * kWideMax + tl[u * kWideMax + j]);
    }
  }
  __device__ __forceinline__ static int ldcg_i(const int32_t* a) { return __ldcg(a); }

  // SwiGLU of every (expert slot, token) pair, one warp per pair and k block of h: h =
  // bf16(silu(gate) * up) from the gate/up partials (each row block: 64 gate rows, then the
  // matching 64 up rows), as B blocks of the slot's down projection.
  __device__ void swiglu_pack(int U) {
    const int* pairs = swiglu_pairs();
    WGeo gr = wgeo(p, K_RTGU, U, gridDim.x);
    wsplit(gr, m, p, K_RTGU, U, gridDim.x);
    const WGeo gs = wgeo(p, K_SHGU, 0, gridDim.x);
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
      const int nc = wn_contrib(g, seg, gridDim.x);
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
      // the slot's j-th token (ascending): rows 2j, 2j + 1
      const int j = __popcll(m->umask[u] & ((1ull << t) - 1ull));
      const size_t blk = (size_t)u * p.kb_i + kb;
      pack4(w.pbh + blk * PBS, w.exh + blk * kWideMax + j, j, lane * 4, f);
    }
  }

  // Layer output of token t: x_mid + the down partials of its routed slots (gate-weighted
  // already) and of the shared expert, rounded to bf16; then the next layer's (or the final)
  // RMSNorm as B blocks.
  __device__ void layer_out(int l, int U) {
    WGeo gd = wgeo(p, K_D, U, gridDim.x);
    wsplit(gd, m, p, K_D, U, gridDim.x);
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
          const int nc = wn_contrib(gd, seg, gridDim.x);
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
    if (DEC_TRACE && blockIdx.x == 0 && tid == 0) p.trace[0] = gtimer();
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
      gather(U);
      gbar();
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
    if (DEC_TRACE && blockIdx.x == 0 && tid == 0) {
      p.trace[kWaitTrace + 4] = tw_prod;
      p.trace[kWaitTrace + 5] = tw_stage;
      p.trace[kWaitTrace + 6] = tw_ld;
      p.trace[kWaitTrace + 7] = tw_flush;
      p.trace[kWaitTrace + 26] = tw_dprod;
      p.trace[kWaitTrace + 27] = tw_dstage;
      p.trace[kWaitTrace + 28] = tw_dflush;
      p.trace[kWaitTrace + 8] = tw_kv;
      p.trace[kWaitTrace + 9] = tw_attn;
      p.trace[kWaitTrace + 10] = tw_pro;
      p.trace[kWaitTrace + 11] = tw_post;
      for (int i = 0; i < 8; ++i) p.trace[kWaitTrace + 12 + i] = tw_a[i];
    }
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
    mbar_init(&m->sbar, 1);
    mbar_init(&m->obar, 1);
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
  WConsumer<NR, HD, G> cons(p, w, ring, full, empty, red, m, reinterpret_cast<float4*>(smem + L.acc_off));
  cons.run();
}

}  // namespace wide
}  // namespace dec
