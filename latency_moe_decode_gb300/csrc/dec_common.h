// Internal layout shared by the engine's host code and its persistent kernel.
#pragma once
#include <cuda.h>  // CUtensorMap

#include <cstdint>

namespace dec {

// Tiles: 128 weight rows x 128 columns of E4M3 codes (one 128x128 scale block), stored in the
// order the consumer warps read them, followed by a 16-byte header {scale of rows 0..63, scale
// of rows 64..127, 0, 0}. Two 64-row halves may come from different matrices (q/k/v heads, or
// an expert's gate and up rows interleaved so one tile yields both SwiGLU operands).
constexpr int kTileRows = 128;
constexpr int kTileK = 128;
constexpr int kTileData = kTileRows * kTileK;  // 16384
constexpr int kTileBytes = kTileData + 16;     // 16400
// One ring slot holds two consecutive weight tiles of a CTA's share (or one KV tile of 64
// positions): each slot is one bulk-copy hand-off, and on this GPU the streaming rate of one SM
// grows with the bytes per hand-off up to ~32 KB (16 KB slots streamed ~4.3 TB/s in total,
// 32 KB slots ~7.0 TB/s).
constexpr int kSlotTiles = 2;
constexpr int kSlotBytes = kSlotTiles * kTileBytes;  // 32800
constexpr int kSlotsInFlight = 2;                     // copies a CTA keeps in flight (at most)
constexpr int kConsumerWarps = 8;
constexpr int kThreads = (kConsumerWarps + 2) * 32;  // + the producer warp and the MMA warp
constexpr int kKvTilePos = 64;                       // KV positions per ring slot
constexpr int kMaxBatch = 8;                         // tokens of one step of decode_step_kernel
constexpr int kWideMax = 64;                         // tokens of one step of the wide kernel (5 .. 64)
constexpr int kMaxHidden = 4096;                     // hidden sizes the kernel handles
constexpr int kTraceSlots = 512;                     // CTA-0 / producer trace words per step
#ifndef DEC_STAMPS
#define DEC_STAMPS 0  // 1: record the per-CTA dependency stamps (diagnostics)
#endif
#ifndef DEC_TRACE
#define DEC_TRACE 0  // 1: record CTA 0's event trace (diagnostics)
#endif
constexpr int kStampsPerLayer = 16;                  // per-CTA dependency time stamps of a layer
constexpr int kStampLayers = 8;                      // layers whose stamps are kept
constexpr int kBarTrace = kStampsPerLayer * kStampLayers;  // per-CTA stamp words per CTA

// Device error codes (low byte) -- the upper bytes carry where it happened.
enum : int {
  kDevOk = 0,
  kDevTimeout = 1,
  kDevBadArg = 2,
  kDevRange = 3,  // an activation outside the f16 range of the CUDA-core GEMV input staging
};

struct LayerDev {
  const uint8_t* qkv;     // tiles, q/k/v rows, [n_rb_qkv][kb_d]
  const uint8_t* o;       // [n_rb_d][kb_o]
  const uint8_t* router;  // [n_rb_router][kb_d]
  const uint8_t* sh_gu;   // shared (or dense FFN) gate/up, [n_rb_gu][kb_d]
  const uint8_t* sh_d;    // shared (or dense FFN) down, [n_rb_d][kb_i]
  const uint8_t* e_gu;    // routed experts gate/up, expert e at e_gu + e * e_gu_stride
  const uint8_t* e_d;     // routed experts down
  const uint16_t* attn_norm;
  const uint16_t* ffn_norm;
};

// Everything the kernel reads, passed by value at launch.
struct KParams {
  // model shape
  int L, d, hq, hkv, hd, E, topk, inter, nsh, dense, V, max_ctx, MB;
  float eps;
  // tile geometry
  int kb_d, kb_o, kb_i;
  int n_rb_qkv, n_rb_d, n_rb_gu, n_rb_router, n_rb_lm;
  long long e_gu_stride, e_d_stride;
  int umax;       // most distinct routed experts one step can select
  int nch;        // attention chunks per (sequence, KV head)
  int ring;       // ring slots
  int inflight;   // most slot copies of one CTA in flight at a time (1..ring)
  int xmax;       // elements per token of the shared-memory activation buffer
  // weights and tables
  const LayerDev* layers;
  const uint16_t* embed;
  const uint16_t* final_norm;
  const uint8_t* lm;
  const uint8_t* warena;  // every repacked weight tile lives in [warena, warena + warena_bytes)
  unsigned long long warena_bytes;
  unsigned long long kv_bytes;  // bytes of each of kc / vc
  const float2* rope;  // [max_ctx][hd/2] (cos, sin)
  uint16_t* kc;        // [L][MB][hkv][max_ctx][hd]
  uint16_t* vc;
  int32_t* lengths;    // [slots]
  int slots;           // KV cache slots (sequences); MB is the token capacity of one step
  int rows;            // max(kMaxBatch, slots): token rows of the routing records and of the
                       // per-step token arrays of a resident generation
  // activations
  uint16_t* xbuf;   // [2][MB][d]
  uint16_t* xmid;   // [MB][d]
  uint16_t* qbuf;   // [MB][hq*hd]
  uint16_t* obuf;   // [MB][hq*hd]
  uint16_t* hsh;    // [MB][inter_sh]
  uint16_t* hrt;    // [umax][MB][inter]
  // split-K partial sums: [segment][slot][MB][128] fp32, and per-output arrival counters
  float *part_qkv, *part_o, *part_router, *part_shgu, *part_rtgu, *part_d, *part_lm;
  // q/k/v and output-projection partials are read directly by the next stage: their counters
  // only grow (one arrival per contributor per launch), [L][row blocks]
  int *cnt_qkv, *cnt_o;
  // router partials: growing counter per layer [L]. Finalised outputs (SwiGLU h, down projection +
  // residual, logits): arrival counters that the group's designated finaliser waits on and resets
  int *cnt_router, *cnt_shgu, *cnt_rtgu, *cnt_d, *cnt_lm, *cnt_lm_done;
  int* o_cnt;  // [L][hkv] merged attention slices written, all sequences (zero between launches)
  unsigned* x_flag;  // [L][n_rb_d] = epoch once a row block of the layer's output is final
  int* h_cnt;  // [L][umax + 1] grows by n_rb_gu per step: an expert slot's SwiGLU row blocks final
                     // (slot umax: the shared / dense expert)
  // attention split-KV partials: [MB][hkv][nch][group][hd + 2], counters [MB][hkv]
  float* attn_part;
  int* attn_cnt;  // [L][MB][hkv] chunk partials published (zero between launches)
  // routing of each layer, written by CTA 0 for inspection (every CTA computes it itself)
  int* rt_idx;        // [L][rows][topk] selections (score-descending)
  float* rt_topk_gate;// [L][rows][topk]
  float* rt_logits;   // [L][rows][E] router logits the selection was made from
  unsigned long long* amax;  // [rows] packed (ordered logit, ~id) maxima
  int* err;           // device status word
  float* logits_ws;   // [MB][V] when the caller gives no logits buffer
  unsigned long long* trace;  // [kTraceSlots + kBarTrace * grid]
  // CTA 0's %globaltimer when the input of layer l was ready (l = 0: step start; l = L: the
  // final norm's input) and, at [L + 1], when CTA 0 finished the step: [L + 2], every build
  unsigned long long* layer_ts;
  int test_skip;  // nonzero only in tests: the first q/k/v tile's arrival of layer 0 is withheld
  // this step
  const int32_t* tokens;
  const uint16_t* hidden_in;
  int B, seq0;
  // 1: the B tokens are consecutive positions length[seq0] .. + B - 1 of slot seq0 (a verify or
  // prefill step), each attending over the cache and the step's earlier new keys (causal)
  int mpos;
  // verify steps: the number of draft tokens accepted (tokens[j + 1] == argmax after position j
  // for j < m) is written here and the slot's length set to length + m + 1
  int32_t* accepted;
  // resident generation: nsteps > 1 decode steps in one launch, step s using epoch + s, reading
  // its tokens at tokens + s * rows and writing the argmax at next_tokens + s * rows; each step's
  // last LM finaliser publishes tok_flag = its epoch once the next tokens are written
  int nsteps;
  unsigned* tok_flag;
  float* logits;
  int32_t* next_tokens;
  uint16_t* hidden_out;
  unsigned epoch;
  unsigned long long timeout_ns;
};

// The wide kernel's own buffers (steps of 5 .. 64 tokens). Every GEMV stage input is kept in
// global memory as the tensor cores' B operand: per k block of 128 activations one block of
// nr rows x 128 bytes (token t's two E4M3 pieces in rows 2t and 2t + 1, canonical K-major layout
// of 8-row x 16-byte core matrices; nr = the kernel's row count, 32, 64 or 128) and one exponent
// byte per token (the pieces encode x * 2^a). The producer copies a tile's block into the ring
// slot beside the weight tile.
struct WideParams {
  // tensor maps of the K and V caches for the attention's tile loads: 3-D (head_dim, position,
  // (layer, slot, KV head) plane), 64 x 64 boxes of bf16, 128-byte swizzle
  CUtensorMap kmap, vmap;
  const uint8_t* pb;  // the B operand arena (pbx, pbo, pbh), for the copies' bounds checks
  unsigned long long pb_bytes;
  uint8_t* pbx;       // [kb_d][nr * 128]: the normalised input of a q/k/v, router, gate/up or LM stage
  uint8_t* pbo;       // [kb_o][nr * 128]: the attention output
  uint8_t* pbh;       // [U + n_shared][kb_i][nr * 128]: the SwiGLU rows of each expert slot (its
                      // tokens in ascending order, compact: the slot's j-th token in rows 2j, 2j + 1)
  uint8_t* pbg;       // [U][kb_d][nr * 128]: pbx's rows of each routed slot's tokens, compact
  int8_t* exx;        // [kb_d][kWideMax] exponents of pbx
  int8_t* exo;        // [kb_o][kWideMax]
  int8_t* exh;        // [U + n_shared][kb_i][kWideMax] (by the slot's token index)
  int8_t* exg;        // [U][kb_d][kWideMax] (by the slot's token index)
  int32_t* sel;       // [kWideMax][topk] this layer's selected experts
  float* selg;        // [kWideMax][topk] and their normalised gates
  unsigned* bar;      // grid barrier counter: zero at launch, + 1 per CTA and barrier
  float* attn_part;   // [MB][hkv][nch][group][hd + 2] chunk states (split context)
  uint16_t* xbuf;     // [MB][d] the layer input (residual stream)
  uint16_t* xmid;     // [MB][d] x + attention output projection
  int nch;            // attention chunks per (sequence, KV head)
  int hmax;           // expert slots pbh / exh hold (at least U + n_shared)
};

}  // namespace dec
