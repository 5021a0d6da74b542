// Host side of the decode engine: validation, weight repacking into kernel tiles, KV cache and
// workspace allocation, the per-step cooperative launch and status readback. Implements dec.h.
#include <cuda_runtime.h>
#include <cudaTypedefs.h>  // PFN_cuTensorMapEncodeTiled

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "dec.h"
#include "dec_kernel.cuh"
#include "dec_wide_host.h"

using namespace dec;

namespace {

// ---------------------------------------------------------------------------------------------
// repacking: a tile is two 64-row halves; each half comes from one source matrix.

struct RepackDesc {
  const uint8_t* w[3];
  const float* s[3];
  int n[3];       // rows of each source
  int halves[3];  // 64-row halves taken from each source (stacked mode)
  int nsrc;
  int interleave; // 1: half h comes from source h % 2, rows 64 * (h / 2)
  int K;          // columns (multiple of 128)
};

__global__ void repack_kernel(const RepackDesc d, uint8_t* dst) {
  const int kbn = d.K / kTileK;
  const int tile = blockIdx.x;  // rb * kbn + kb
  const int rb = tile / kbn, kb = tile % kbn;
  uint8_t* out = dst + (size_t)tile * kTileBytes;
  for (int q = threadIdx.x; q < kTileData / 16; q += blockDim.x) {
    // the tensor cores' canonical K-major layout without swizzling: 16-byte chunk c of tile row
    // 8g + r sits at unit (8g + c) * 8 + r (core matrices of 8 rows x 16 bytes, 128 bytes apart
    // along K, 1024 bytes apart along the rows)
    const int r = q & 7, c = (q >> 3) & 7, g8 = q >> 6;
    const int row = g8 * 8 + r;  // row inside the tile
    const int h = rb * 2 + row / 64;
    int src = -1, srow = 0;
    if (d.interleave) {
      src = h & 1;
      srow = (h >> 1) * 64 + (row & 63);
    } else {
      int hh = h;
      for (int s = 0; s < d.nsrc; ++s) {
        if (hh < d.halves[s]) {
          src = s;
          srow = hh * 64 + (row & 63);
          break;
        }
        hh -= d.halves[s];
      }
    }
    uint4 v = make_uint4(0, 0, 0, 0);
    if (src >= 0 && srow < d.n[src]) {
      const uint8_t* p = d.w[src] + (size_t)srow * d.K + kb * kTileK + c * 16;
      v = *reinterpret_cast<const uint4*>(p);
    }
    *reinterpret_cast<uint4*>(out + (size_t)q * 16) = v;
  }
  if (threadIdx.x < 2) {
    const int h = rb * 2 + threadIdx.x;
    int src = -1, srow = 0;
    if (d.interleave) {
      src = h & 1;
      srow = (h >> 1) * 64;
    } else {
      int hh = h;
      for (int s = 0; s < d.nsrc; ++s) {
        if (hh < d.halves[s]) {
          src = s;
          srow = hh * 64;
          break;
        }
        hh -= d.halves[s];
      }
    }
    float sc = 0.f;
    if (src >= 0 && srow < d.n[src]) sc = d.s[src][(size_t)(srow / 128) * kbn + kb];
    reinterpret_cast<float*>(out + kTileData)[threadIdx.x] = sc;
    if (threadIdx.x == 0) reinterpret_cast<float*>(out + kTileData)[2] = 0.f;
    if (threadIdx.x == 1) reinterpret_cast<float*>(out + kTileData)[3] = 0.f;
  }
}

__global__ void transpose_tokens_kernel(const int32_t* src, int n_seq, int n_tok, int32_t* dst) {
  int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n_seq * n_tok) {
    int s = i / n_tok, t = i % n_tok;
    dst[(size_t)t * n_seq + s] = src[i];
  }
}

// ---------------------------------------------------------------------------------------------

using KernelFn = void (*)(const KParams);

template <int BM, int HD, int G>
KernelFn pick_kernel() {
  return decode_step_kernel<BM, HD, G>;
}

KernelFn kernel_for(int bm, int hd, int group) {
#define DEC_K(B, H, GR) \
  if (bm == B && hd == H && group == GR) return pick_kernel<B, H, GR>();
  DEC_K(1, 64, 2) DEC_K(2, 64, 2) DEC_K(4, 64, 2) DEC_K(8, 64, 2)
  DEC_K(1, 128, 4) DEC_K(2, 128, 4) DEC_K(4, 128, 4) DEC_K(8, 128, 4)
#undef DEC_K
  return nullptr;
}

const int kBmChoices[4] = {1, 2, 4, 8};

}  // namespace

struct dec_engine {
  dec_model_cfg cfg{};
  int device = 0, sms = 0, grid = 0;
  cudaStream_t stream = nullptr;
  // The stream of the engine's most recent work. Consecutive steps share counters, exchange
  // buffers and the KV cache, so work on another stream is ordered after it (order_on).
  cudaStream_t last_stream = nullptr;
  cudaEvent_t order_ev = nullptr;
  KParams base{};
  std::vector<void*> allocs;
  LayerDev* d_layers = nullptr;
  int hd = 0, group = 0;
  KernelFn kern[4] = {nullptr, nullptr, nullptr, nullptr};
  int smem[4] = {0, 0, 0, 0};
  int ring[4] = {0, 0, 0, 0};
  int nch_max = 1;
  int rows = kMaxBatch;  // max(kMaxBatch, max_batch): routing records and per-step token rows
  // steps of more than kMaxBatch tokens: the wide kernels (B operand blocks of 32, 64, 128 rows
  // for up to 16, 32, 64 tokens), their parameters and buffers
  KParams wbase{};
  WideParams wp{};
  wide::WideKernelFn wkern[3] = {nullptr, nullptr, nullptr};
  int wsmem[3] = {0, 0, 0}, wring[3] = {0, 0, 0};
  int wnch_max = 1;
  int winflight = 4;  // copies one CTA of the wide kernel keeps in flight (DEC_WIDE_INFLIGHT)
  int inflight = kSlotsInFlight;  // the same for decode_step_kernel (DEC_INFLIGHT)
  // decode steps of at least this many tokens take the wide kernel (measured at 1k context on
  // the 8-layer stack: 8 tokens 3921 vs 3313 tokens/s on decode_step_kernel, 4 tokens 2494 vs
  // 2663, 2 tokens 1525 vs 2001)
  int wide_min = wide::kWideMinBatch;
  std::vector<int32_t> lengths;
  unsigned epoch = 0;
  // Counters that grow across steps (each arrival adds its tile count, at most kbs per row block
  // and step) and flags that hold the step's epoch. They are zeroed and the epoch restarts at 1
  // before a counter could leave the int range.
  unsigned epoch_limit = 0;
  std::vector<std::pair<void*, size_t>> epoch_bufs;
  bool poisoned = false;
  std::string err;
  int32_t* d_hist = nullptr;
  int32_t* d_accepted = nullptr;  // verify steps: the accepted draft count
  int64_t launches = 0, weight_bytes = 0, kv_bytes = 0, ws_bytes = 0;
  uint8_t* arena = nullptr;  // all repacked weight tiles (one allocation the kernel bounds-checks)
  size_t arena_size = 0, arena_used = 0;
};

namespace {

dec_status fail(dec_engine* e, dec_status s, const std::string& msg);

// Tensor map of one KV cache (kc or vc: [layer][slot][KV head][position][head_dim] bf16) for the
// wide kernel's tile loads: 3-D (head_dim, position, (layer, slot, KV head) plane), boxes of 64
// values x 64 positions in the 128-byte swizzled layout, zeros past the cache's end.
dec_status encode_kv_map(dec_engine* e, CUtensorMap* map, void* base, const dec_model_cfg& c) {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
  cudaError_t ce = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
  if (ce != cudaSuccess || q != cudaDriverEntryPointSuccess || fn == nullptr)
    return fail(e, DEC_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
  const cuuint64_t dims[3] = {(cuuint64_t)c.head_dim, (cuuint64_t)c.max_ctx,
                              (cuuint64_t)c.n_layers * c.max_batch * c.n_kv_heads};
  const cuuint64_t strides[2] = {(cuuint64_t)c.head_dim * 2, (cuuint64_t)c.max_ctx * c.head_dim * 2};
  const cuuint32_t box[3] = {64, 64, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn)(
      map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
      CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(e, DEC_ERR_CUDA, "cuTensorMapEncodeTiled failed (" + std::to_string((int)r) + ")");
  return DEC_OK;
}

dec_status fail(dec_engine* e, dec_status s, const std::string& msg) {
  if (e) e->err = msg;
  return s;
}

dec_status cuda_fail(dec_engine* e, cudaError_t c, const char* what) {
  return fail(e, c == cudaErrorMemoryAllocation ? DEC_ERR_OOM : DEC_ERR_CUDA,
              std::string(what) + ": " + cudaGetErrorString(c));
}

#define DEC_CUDA(call)                                   \
  do {                                                   \
    cudaError_t _c = (call);                             \
    if (_c != cudaSuccess) return cuda_fail(e, _c, #call); \
  } while (0)

template <typename T>
dec_status dalloc(dec_engine* e, T** p, size_t bytes, int64_t* account) {
  void* v = nullptr;
  cudaError_t c = cudaMalloc(&v, bytes ? bytes : 16);
  if (c != cudaSuccess) return cuda_fail(e, c, "cudaMalloc");
  e->allocs.push_back(v);
  if (account) *account += (int64_t)bytes;
  *p = reinterpret_cast<T*>(v);
  return DEC_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

dec_status carve(dec_engine* e, size_t bytes, uint8_t** out) {
  const size_t at = (e->arena_used + 255) & ~(size_t)255;
  if (at + bytes > e->arena_size) return fail(e, DEC_ERR_ARG, "weight arena overflow");
  *out = e->arena + at;
  e->arena_used = at + bytes;
  e->weight_bytes += (int64_t)bytes;
  return DEC_OK;
}

dec_status repack(dec_engine* e, const RepackDesc& d, int n_rb, uint8_t** out) {
  for (int s = 0; s < d.nsrc; ++s)
    if (d.w[s] && (!aligned16(d.w[s]) || !d.s[s])) return fail(e, DEC_ERR_ARG, "weight not 16-byte aligned or scale missing");
  const int kbn = d.K / kTileK;
  size_t bytes = (size_t)n_rb * kbn * kTileBytes;
  dec_status st = carve(e, bytes, out);
  if (st != DEC_OK) return st;
  repack_kernel<<<n_rb * kbn, 256, 0, e->stream>>>(d, *out);
  DEC_CUDA(cudaGetLastError());
  return DEC_OK;
}

RepackDesc plain_desc(const dec_fp8_mat& m, int n, int K) {
  RepackDesc d{};
  d.w[0] = static_cast<const uint8_t*>(m.w);
  d.s[0] = m.scale;
  d.n[0] = n;
  d.halves[0] = (n + 63) / 64;
  d.nsrc = 1;
  d.K = K;
  return d;
}

RepackDesc gu_desc(const dec_fp8_mat& g, const dec_fp8_mat& u, int inter, int K) {
  RepackDesc d{};
  d.w[0] = static_cast<const uint8_t*>(g.w);
  d.s[0] = g.scale;
  d.n[0] = inter;
  d.w[1] = static_cast<const uint8_t*>(u.w);
  d.s[1] = u.scale;
  d.n[1] = inter;
  d.nsrc = 2;
  d.interleave = 1;
  d.K = K;
  return d;
}

dec_status copy_bf16(dec_engine* e, const void* src, size_t n, uint16_t** out) {
  dec_status st = dalloc(e, out, n * 2, &e->weight_bytes);
  if (st != DEC_OK) return st;
  if (!src) return fail(e, DEC_ERR_ARG, "missing bf16 tensor");
  DEC_CUDA(cudaMemcpyAsync(*out, src, n * 2, cudaMemcpyDeviceToDevice, e->stream));
  return DEC_OK;
}

int range_lo_h(int T, int c, int G) { return (int)((long long)T * c / G); }

// Order work about to be queued on stream s after everything the engine queued before (on
// whichever stream that was): an event on the previous stream that s waits for, only when the
// stream changes. Steps of one engine therefore never overlap, whatever streams they are given.
dec_status order_on(dec_engine* e, cudaStream_t s) {
  if (e->last_stream != s) {
    DEC_CUDA(cudaEventRecord(e->order_ev, e->last_stream));
    DEC_CUDA(cudaStreamWaitEvent(s, e->order_ev, 0));
    e->last_stream = s;
  }
  return DEC_OK;
}

// Wait on the host for all of the engine's queued work (and nothing else on the device).
dec_status quiesce(dec_engine* e) {
  dec_status st = order_on(e, e->stream);
  if (st != DEC_OK) return st;
  DEC_CUDA(cudaStreamSynchronize(e->stream));
  return DEC_OK;
}

// Entry points that queue work need the engine's device to be the current one.
dec_status check_device(dec_engine* e) {
  int cur = -1;
  DEC_CUDA(cudaGetDevice(&cur));
  if (cur != e->device) return fail(e, DEC_ERR_ARG, "the engine's device is not the current CUDA device");
  return DEC_OK;
}

dec_status check_device_status(dec_engine* e) {
  int code = 0;
  DEC_CUDA(cudaMemcpyAsync(&code, e->base.err, sizeof(int), cudaMemcpyDeviceToHost, e->stream));
  DEC_CUDA(cudaStreamSynchronize(e->stream));
  if (code == 0) return DEC_OK;
  e->poisoned = true;
  char buf[160];
  const int kind = code & 0xFF, where = code >> 8;
  if (kind == kDevTimeout) {
    snprintf(buf, sizeof buf, "device wait timed out (site %d); engine poisoned", where);
    return fail(e, DEC_ERR_TIMEOUT, buf);
  }
  if (kind == kDevRange) {
    snprintf(buf, sizeof buf, "an activation left the f16 staging range (site %d); engine poisoned", where);
    return fail(e, DEC_ERR_DEVICE, buf);
  }
  snprintf(buf, sizeof buf, "device check failed (code %d, site %d); engine poisoned", kind, where);
  return fail(e, DEC_ERR_DEVICE, buf);
}

}  // namespace

// Staging for dec_prefill_kv_noalloc: the step-major token ids of one token-mode prefill, one copy
// per device (a file-scope device array, so that entry point allocates no device memory).
static __device__ __align__(256) int32_t g_prefill_ids[DEC_NOALLOC_PREFILL_MAX_IDS];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_prefill_ids_mu;
int32_t* g_prefill_ids_addr[kMaxDevices] = {};

// Device address of the engine's device's copy of g_prefill_ids. Looked up once per device, with
// that device current, then cached; the caller's current device is restored.
dec_status prefill_ids_scratch(dec_engine* e, int32_t** out) {
  if (e->device < 0 || e->device >= kMaxDevices)
    return fail(e, DEC_ERR_UNSUPPORTED, "device ordinal beyond the static scratch table");
  std::lock_guard<std::mutex> lock(g_prefill_ids_mu);
  if (!g_prefill_ids_addr[e->device]) {
    int cur = -1;
    cudaError_t ce = cudaGetDevice(&cur);
    if (ce != cudaSuccess) return cuda_fail(e, ce, "cudaGetDevice");
    if (cur != e->device) {
      ce = cudaSetDevice(e->device);
      if (ce != cudaSuccess) return cuda_fail(e, ce, "cudaSetDevice");
    }
    void* addr = nullptr;
    ce = cudaGetSymbolAddress(&addr, g_prefill_ids);
    if (cur != e->device) {
      cudaError_t back = cudaSetDevice(cur);
      if (ce == cudaSuccess && back != cudaSuccess) return cuda_fail(e, back, "cudaSetDevice (restore)");
    }
    if (ce != cudaSuccess) return cuda_fail(e, ce, "cudaGetSymbolAddress");
    if (!addr) return fail(e, DEC_ERR_CUDA, "cudaGetSymbolAddress returned a null address");
    g_prefill_ids_addr[e->device] = static_cast<int32_t*>(addr);
  }
  *out = g_prefill_ids_addr[e->device];
  return DEC_OK;
}

}  // namespace

extern "C" {

const char* dec_status_string(dec_status s) {
  switch (s) {
    case DEC_OK: return "ok";
    case DEC_ERR_ARG: return "bad argument";
    case DEC_ERR_CUDA: return "CUDA error";
    case DEC_ERR_OOM: return "out of device memory";
    case DEC_ERR_TIMEOUT: return "device wait timed out";
    case DEC_ERR_UNSUPPORTED: return "unsupported shape";
    case DEC_ERR_POISONED: return "engine poisoned by an earlier device error";
    case DEC_ERR_DEVICE: return "device-side check failed";
    case DEC_ERR_CAPACITY: return "sequence would exceed max_ctx";
  }
  return "unknown status";
}

dec_status dec_validate_cfg(const dec_model_cfg* c) {
  if (!c) return DEC_ERR_ARG;
  if (c->n_layers < 1 || c->hidden < 1 || c->n_heads < 1 || c->n_kv_heads < 1 || c->head_dim < 1 ||
      c->max_ctx < 1 || c->max_batch < 1 || c->vocab < 0 || c->n_experts < 0 || c->dense_ffn < 0 ||
      c->n_shared < 0 || !(c->rms_eps >= 0.f) || !(c->rope_theta > 0.f))
    return DEC_ERR_ARG;
  if (c->n_heads % c->n_kv_heads != 0) return DEC_ERR_ARG;
  if ((c->n_experts > 0) == (c->dense_ffn > 0)) return DEC_ERR_ARG;  // exactly one FFN kind
  if (c->n_experts > 0 && (c->top_k < 1 || c->top_k > c->n_experts || c->moe_inter < 1)) return DEC_ERR_ARG;
  if (c->head_dim % 2 != 0) return DEC_ERR_ARG;
  // implemented subset
  const int group = c->n_heads / c->n_kv_heads;
  if (!((c->head_dim == 64 && group == 2) || (c->head_dim == 128 && group == 4))) return DEC_ERR_UNSUPPORTED;
  if (c->hidden % 128 != 0 || (c->n_heads * c->head_dim) % 128 != 0) return DEC_ERR_UNSUPPORTED;
  if (c->n_experts > 0) {
    if (c->n_experts > kMaxExperts || c->top_k > 16 || c->moe_inter % 128 != 0 || c->n_shared > 1)
      return DEC_ERR_UNSUPPORTED;
  } else if (c->dense_ffn % 128 != 0) {
    return DEC_ERR_UNSUPPORTED;
  }
  if (c->max_batch > kWideMax || c->n_kv_heads > 64 || c->hidden > kMaxHidden) return DEC_ERR_UNSUPPORTED;
  // decode batches above 8 (the wide kernel) hold at most 8 experts per token
  if (c->max_batch > kMaxBatch && c->n_experts > 0 && c->top_k > wide::kWideTopkHost) return DEC_ERR_UNSUPPORTED;
  return DEC_OK;
}

dec_status dec_init(const dec_model_cfg* cfg, const dec_weights* W, void* stream, dec_engine** out) {
  if (!out) return DEC_ERR_ARG;
  *out = nullptr;
  dec_status vs = dec_validate_cfg(cfg);
  if (vs != DEC_OK) return vs;
  if (!W || !W->layers) return DEC_ERR_ARG;
  if (cfg->vocab > 0 && (!W->embed || !W->final_norm || !W->lm_head.w)) return DEC_ERR_ARG;

  dec_engine* e = new dec_engine();
  e->cfg = *cfg;
  const dec_model_cfg& c = *cfg;
  dec_status st = DEC_OK;
  auto bail = [&](dec_status s) {
    dec_destroy(e);
    return s;
  };

  cudaError_t ce = cudaGetDevice(&e->device);
  if (ce != cudaSuccess) return bail(cuda_fail(e, ce, "cudaGetDevice"));
  cudaDeviceProp prop;
  ce = cudaGetDeviceProperties(&prop, e->device);
  if (ce != cudaSuccess) return bail(cuda_fail(e, ce, "cudaGetDeviceProperties"));
  e->sms = prop.multiProcessorCount;
  if (!prop.cooperativeLaunch) return bail(DEC_ERR_UNSUPPORTED);
  ce = cudaStreamCreateWithFlags(&e->stream, cudaStreamNonBlocking);
  if (ce != cudaSuccess) return bail(cuda_fail(e, ce, "cudaStreamCreate"));
  e->last_stream = e->stream;
  ce = cudaEventCreateWithFlags(&e->order_ev, cudaEventDisableTiming);
  if (ce != cudaSuccess) return bail(cuda_fail(e, ce, "cudaEventCreate"));
  cudaStream_t user = stream ? static_cast<cudaStream_t>(stream) : e->stream;
  // weights are read on the engine's stream: order after the caller's pending work
  {
    cudaEvent_t ev;
    cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
    cudaEventRecord(ev, user);
    cudaStreamWaitEvent(e->stream, ev, 0);
    cudaEventDestroy(ev);
  }

  KParams& p = e->base;
  const bool dense = c.dense_ffn > 0;
  e->hd = c.head_dim;
  e->group = c.n_heads / c.n_kv_heads;
  p.L = c.n_layers;
  p.d = c.hidden;
  p.hq = c.n_heads;
  p.hkv = c.n_kv_heads;
  p.hd = c.head_dim;
  p.E = dense ? 0 : c.n_experts;
  p.topk = dense ? 0 : c.top_k;
  p.inter = dense ? c.dense_ffn : c.moe_inter;
  p.nsh = dense ? 1 : c.n_shared;
  p.dense = dense ? 1 : 0;
  p.V = c.vocab;
  p.max_ctx = c.max_ctx;
  p.MB = kMaxBatch;  // tokens one step can take: sequences side by side, or positions of one
  p.slots = c.max_batch;
  e->rows = std::max(kMaxBatch, c.max_batch);
  p.rows = e->rows;
  p.eps = c.rms_eps;
  p.kb_d = c.hidden / kTileK;
  p.kb_o = c.n_heads * c.head_dim / kTileK;
  p.kb_i = p.inter / kTileK;
  p.n_rb_qkv = ((c.n_heads + 2 * c.n_kv_heads) * c.head_dim + kTileRows - 1) / kTileRows;
  p.n_rb_d = c.hidden / kTileRows;
  p.n_rb_gu = p.inter / 64;
  p.n_rb_router = dense ? 0 : (c.n_experts + kTileRows - 1) / kTileRows;
  p.n_rb_lm = (c.vocab + kTileRows - 1) / kTileRows;
  p.e_gu_stride = (long long)p.n_rb_gu * p.kb_d * kTileBytes;
  p.e_d_stride = (long long)p.n_rb_d * p.kb_i * kTileBytes;
  p.umax = dense ? 0 : std::min(c.n_experts, p.MB * c.top_k);
  e->grid = e->sms;
  const int G = e->grid;
  {
    // the kernel's tile-ownership arithmetic is 32-bit: (tiles of a stage + 1) x grid < 2^31
    const long long t_max = std::max({(long long)p.n_rb_lm * p.kb_d, (long long)p.n_rb_qkv * p.kb_d,
                                      (long long)(p.umax + p.nsh) * p.n_rb_d * p.kb_i,
                                      (long long)std::max(1, p.umax) * p.n_rb_gu * p.kb_d});
    if ((t_max + 1) * G >= (1LL << 31)) return bail(fail(e, DEC_ERR_UNSUPPORTED, "too many tiles in one stage"));
  }

  // ---- weights: one arena for every repacked tile
  {
    const size_t TB = kTileBytes;
    size_t per_layer = (size_t)p.n_rb_qkv * p.kb_d + (size_t)p.n_rb_d * p.kb_o;
    if (dense) {
      per_layer += (size_t)p.n_rb_gu * p.kb_d + (size_t)p.n_rb_d * p.kb_i;
    } else {
      per_layer += (size_t)p.n_rb_router * p.kb_d;
      per_layer += (size_t)(c.n_shared + c.n_experts) * ((size_t)p.n_rb_gu * p.kb_d + (size_t)p.n_rb_d * p.kb_i);
    }
    e->arena_size = per_layer * TB * c.n_layers + (size_t)p.n_rb_lm * p.kb_d * TB + 256 * (16 * (size_t)c.n_layers + 16);
    if ((st = dalloc(e, &e->arena, e->arena_size, nullptr)) != DEC_OK) return bail(st);
    p.warena = e->arena;
    p.warena_bytes = e->arena_size;
  }
  std::vector<LayerDev> layers(c.n_layers);
  for (int l = 0; l < c.n_layers; ++l) {
    const dec_layer_weights& Lw = W->layers[l];
    LayerDev& Ld = layers[l];
    RepackDesc q{};
    q.w[0] = static_cast<const uint8_t*>(Lw.wq.w);
    q.s[0] = Lw.wq.scale;
    q.n[0] = c.n_heads * c.head_dim;
    q.halves[0] = q.n[0] / 64;
    q.w[1] = static_cast<const uint8_t*>(Lw.wk.w);
    q.s[1] = Lw.wk.scale;
    q.n[1] = c.n_kv_heads * c.head_dim;
    q.halves[1] = q.n[1] / 64;
    q.w[2] = static_cast<const uint8_t*>(Lw.wv.w);
    q.s[2] = Lw.wv.scale;
    q.n[2] = c.n_kv_heads * c.head_dim;
    q.halves[2] = q.n[2] / 64;
    q.nsrc = 3;
    q.K = c.hidden;
    if (!q.w[0] || !q.w[1] || !q.w[2] || !Lw.wo.w || !Lw.attn_norm || !Lw.ffn_norm)
      return bail(fail(e, DEC_ERR_ARG, "missing attention weights"));
    uint8_t* t = nullptr;
    if ((st = repack(e, q, p.n_rb_qkv, &t)) != DEC_OK) return bail(st);
    Ld.qkv = t;
    if ((st = repack(e, plain_desc(Lw.wo, c.hidden, c.n_heads * c.head_dim), p.n_rb_d, &t)) != DEC_OK) return bail(st);
    Ld.o = t;
    uint16_t* nb = nullptr;
    if ((st = copy_bf16(e, Lw.attn_norm, c.hidden, &nb)) != DEC_OK) return bail(st);
    Ld.attn_norm = nb;
    if ((st = copy_bf16(e, Lw.ffn_norm, c.hidden, &nb)) != DEC_OK) return bail(st);
    Ld.ffn_norm = nb;
    if (dense) {
      if (!Lw.ffn_gate.w || !Lw.ffn_up.w || !Lw.ffn_down.w) return bail(fail(e, DEC_ERR_ARG, "missing FFN weights"));
      if ((st = repack(e, gu_desc(Lw.ffn_gate, Lw.ffn_up, p.inter, c.hidden), p.n_rb_gu, &t)) != DEC_OK) return bail(st);
      Ld.sh_gu = t;
      if ((st = repack(e, plain_desc(Lw.ffn_down, c.hidden, p.inter), p.n_rb_d, &t)) != DEC_OK) return bail(st);
      Ld.sh_d = t;
    } else {
      if (!Lw.router.w || !Lw.expert_gate || !Lw.expert_up || !Lw.expert_down ||
          (c.n_shared > 0 && (!Lw.shared_gate || !Lw.shared_up || !Lw.shared_down)))
        return bail(fail(e, DEC_ERR_ARG, "missing MoE weights"));
      if ((st = repack(e, plain_desc(Lw.router, c.n_experts, c.hidden), p.n_rb_router, &t)) != DEC_OK) return bail(st);
      Ld.router = t;
      if (c.n_shared > 0) {
        if ((st = repack(e, gu_desc(Lw.shared_gate[0], Lw.shared_up[0], p.inter, c.hidden), p.n_rb_gu, &t)) != DEC_OK)
          return bail(st);
        Ld.sh_gu = t;
        if ((st = repack(e, plain_desc(Lw.shared_down[0], c.hidden, p.inter), p.n_rb_d, &t)) != DEC_OK) return bail(st);
        Ld.sh_d = t;
      }
      uint8_t* egu = nullptr;
      uint8_t* ed = nullptr;
      if ((st = carve(e, (size_t)c.n_experts * p.e_gu_stride, &egu)) != DEC_OK) return bail(st);
      if ((st = carve(e, (size_t)c.n_experts * p.e_d_stride, &ed)) != DEC_OK) return bail(st);
      for (int x = 0; x < c.n_experts; ++x) {
        RepackDesc gd = gu_desc(Lw.expert_gate[x], Lw.expert_up[x], p.inter, c.hidden);
        RepackDesc dd = plain_desc(Lw.expert_down[x], c.hidden, p.inter);
        for (int s = 0; s < 2; ++s)
          if (!gd.w[s] || !aligned16(gd.w[s]) || !gd.s[s]) return bail(fail(e, DEC_ERR_ARG, "bad expert weight"));
        if (!dd.w[0] || !aligned16(dd.w[0]) || !dd.s[0]) return bail(fail(e, DEC_ERR_ARG, "bad expert weight"));
        repack_kernel<<<p.n_rb_gu * p.kb_d, 256, 0, e->stream>>>(gd, egu + (size_t)x * p.e_gu_stride);
        repack_kernel<<<p.n_rb_d * p.kb_i, 256, 0, e->stream>>>(dd, ed + (size_t)x * p.e_d_stride);
      }
      ce = cudaGetLastError();
      if (ce != cudaSuccess) return bail(cuda_fail(e, ce, "repack"));
      Ld.e_gu = egu;
      Ld.e_d = ed;
    }
  }
  if ((st = dalloc(e, &e->d_layers, sizeof(LayerDev) * c.n_layers, nullptr)) != DEC_OK) return bail(st);
  ce = cudaMemcpyAsync(e->d_layers, layers.data(), sizeof(LayerDev) * c.n_layers, cudaMemcpyHostToDevice, e->stream);
  if (ce != cudaSuccess) return bail(cuda_fail(e, ce, "copy layers"));
  p.layers = e->d_layers;
  if (c.vocab > 0) {
    uint16_t* emb = nullptr;
    if ((st = copy_bf16(e, W->embed, (size_t)c.vocab * c.hidden, &emb)) != DEC_OK) return bail(st);
    p.embed = emb;
    uint16_t* fn = nullptr;
    if ((st = copy_bf16(e, W->final_norm, c.hidden, &fn)) != DEC_OK) return bail(st);
    p.final_norm = fn;
    uint8_t* t = nullptr;
    if ((st = repack(e, plain_desc(W->lm_head, c.vocab, c.hidden), p.n_rb_lm, &t)) != DEC_OK) return bail(st);
    p.lm = t;
  }

  // ---- RoPE table: angles pos * theta^(-2i/hd) in double, stored as fp32 (cos, sin)
  {
    const int half = c.head_dim / 2;
    std::vector<float2> tab((size_t)c.max_ctx * half);
    for (int pos = 0; pos < c.max_ctx; ++pos)
      for (int i = 0; i < half; ++i) {
        double inv = std::pow((double)c.rope_theta, -2.0 * i / (double)c.head_dim);
        double a = (double)pos * inv;
        tab[(size_t)pos * half + i] = make_float2((float)std::cos(a), (float)std::sin(a));
      }
    float2* d = nullptr;
    if ((st = dalloc(e, &d, tab.size() * sizeof(float2), &e->ws_bytes)) != DEC_OK) return bail(st);
    ce = cudaMemcpy(d, tab.data(), tab.size() * sizeof(float2), cudaMemcpyHostToDevice);
    if (ce != cudaSuccess) return bail(cuda_fail(e, ce, "copy rope"));
    p.rope = d;
  }

  // ---- KV cache
  {
    size_t n = (size_t)c.n_layers * c.max_batch * c.n_kv_heads * c.max_ctx * c.head_dim;
    p.kv_bytes = n * 2;
    if ((st = dalloc(e, &p.kc, n * 2, &e->kv_bytes)) != DEC_OK) return bail(st);
    if ((st = dalloc(e, &p.vc, n * 2, &e->kv_bytes)) != DEC_OK) return bail(st);
    cudaMemsetAsync(p.kc, 0, n * 2, e->stream);
    cudaMemsetAsync(p.vc, 0, n * 2, e->stream);
  }

  // ---- workspace
  {
    const int MB = p.MB, d = c.hidden, qd = c.n_heads * c.head_dim;
    const size_t rows = kTileRows;
    auto zalloc = [&](auto** ptr, size_t bytes) -> dec_status {
      dec_status s2 = dalloc(e, ptr, bytes, &e->ws_bytes);
      if (s2 == DEC_OK && cudaMemsetAsync(*ptr, 0, bytes ? bytes : 16, e->stream) != cudaSuccess) s2 = DEC_ERR_CUDA;
      return s2;
    };
#define Z(ptr, bytes) \
  if ((st = zalloc(&(ptr), (bytes))) != DEC_OK) return bail(st);
    Z(p.lengths, sizeof(int32_t) * c.max_batch);
    Z(e->d_accepted, sizeof(int32_t) * 4);
    Z(p.xbuf, 2ull * MB * d * 2);
    Z(p.xmid, (size_t)MB * d * 2);
    Z(p.qbuf, (size_t)MB * qd * 2);
    Z(p.obuf, (size_t)MB * qd * 2);
    Z(p.hsh, (size_t)MB * p.inter * 2);
    Z(p.hrt, (size_t)std::max(1, p.umax) * MB * p.inter * 2);
    const size_t fb = sizeof(float) * MB * rows;
    Z(p.part_qkv, fb * p.n_rb_qkv * p.kb_d);
    Z(p.part_o, fb * p.n_rb_d * p.kb_o);
    Z(p.part_router, fb * std::max(1, p.n_rb_router) * p.kb_d);
    Z(p.part_shgu, fb * p.n_rb_gu * p.kb_d);
    Z(p.part_rtgu, fb * std::max(1, p.umax) * p.n_rb_gu * p.kb_d);
    Z(p.part_d, fb * (size_t)(p.umax + p.nsh) * p.n_rb_d * p.kb_i);
    Z(p.part_lm, fb * std::max(1, p.n_rb_lm) * p.kb_d);
    Z(p.cnt_qkv, sizeof(int) * (size_t)c.n_layers * p.n_rb_qkv);
    Z(p.cnt_o, sizeof(int) * (size_t)c.n_layers * p.n_rb_d);
    Z(p.o_cnt, sizeof(int) * (size_t)c.n_layers * c.n_kv_heads);
    Z(p.x_flag, sizeof(unsigned) * (size_t)c.n_layers * p.n_rb_d);
    Z(p.h_cnt, sizeof(int) * (size_t)c.n_layers * (p.umax + 1));
    Z(p.cnt_router, sizeof(int) * c.n_layers);
    e->epoch_bufs = {{p.cnt_qkv, sizeof(int) * (size_t)c.n_layers * p.n_rb_qkv},
                     {p.cnt_o, sizeof(int) * (size_t)c.n_layers * p.n_rb_d},
                     {p.cnt_router, sizeof(int) * c.n_layers},
                     {p.x_flag, sizeof(unsigned) * (size_t)c.n_layers * p.n_rb_d},
                     {p.h_cnt, sizeof(int) * (size_t)c.n_layers * (p.umax + 1)}};
    Z(p.cnt_shgu, sizeof(int) * p.n_rb_gu);
    Z(p.cnt_rtgu, sizeof(int) * std::max(1, p.umax) * p.n_rb_gu);
    Z(p.cnt_d, sizeof(int) * p.n_rb_d);
    Z(p.cnt_lm, sizeof(int) * std::max(1, p.n_rb_lm));
    Z(p.cnt_lm_done, sizeof(int) * 32);
    e->nch_max = std::max(1, G / c.n_kv_heads);
    Z(p.attn_part, sizeof(float) * MB * c.n_kv_heads * e->nch_max * e->group * (c.head_dim + 2));
    Z(p.attn_cnt, sizeof(int) * (size_t)c.n_layers * MB * c.n_kv_heads);
    // per step a growing counter gains at most max(kb_d, kb_o, n_rb_gu)
    e->epoch_limit = (1u << 30) / (unsigned)std::max({p.kb_d, p.kb_o, p.n_rb_gu, 1});
    if (const char* el = getenv("DEC_EPOCH_LIMIT")) {  // a smaller limit, for testing the restart
      const long v = atol(el);
      if (v >= 1 && (unsigned long)v < e->epoch_limit) e->epoch_limit = (unsigned)v;
    }
    const size_t RW = (size_t)e->rows;
    Z(p.rt_idx, sizeof(int) * c.n_layers * RW * std::max(1, c.top_k));
    Z(p.rt_topk_gate, sizeof(float) * c.n_layers * RW * std::max(1, c.top_k));
    Z(p.rt_logits, sizeof(float) * c.n_layers * RW * std::max(1, c.n_experts));
    Z(p.amax, sizeof(unsigned long long) * RW);
    Z(p.err, sizeof(int) * 32);
    Z(p.logits_ws, sizeof(float) * RW * std::max(1, c.vocab));
    Z(p.trace, sizeof(unsigned long long) * (kTraceSlots + (size_t)kBarTrace * G));
    Z(p.layer_ts, sizeof(unsigned long long) * (c.n_layers + 2));
    Z(p.tok_flag, sizeof(unsigned) * 32);
    e->epoch_bufs.push_back({p.tok_flag, sizeof(unsigned) * 32});
    p.nsteps = 1;
    Z(e->d_hist, sizeof(int32_t) * (size_t)(c.max_ctx + 1) * RW);
#undef Z
  }

  // ---- activation buffer width: d, n_heads*head_dim, or the experts a CTA's down range spans
  // (down tiles come in runs of one expert slot: kb_i tiles row-block major for at most
  // kDRowMajorMax slots, run s belonging to slot s % nv; otherwise n_rb_d * kb_i tiles, one per slot)
  {
    int xmax = std::max(c.hidden, c.n_heads * c.head_dim);
    int span = 1;
    for (int U = 0; U <= p.umax; ++U) {
      const int nv = U + p.nsh;
      const int T = p.n_rb_d * nv * p.kb_i;
      const int run = nv <= kDRowMajorMax ? p.kb_i : p.n_rb_d * p.kb_i;
      for (int cta = 0; cta < G; ++cta) {
        int t0 = range_lo_h(T, cta, G), t1 = range_lo_h(T, cta + 1, G);
        if (t1 > t0) span = std::max(span, std::min((t1 - 1) / run - t0 / run + 1, nv));
      }
    }
    xmax = std::max(xmax, span * p.inter);
    if (xmax > kMaxKb * kTileK) return bail(fail(e, DEC_ERR_UNSUPPORTED, "a stage input wider than the B operand table"));
    p.xmax = xmax;
  }

  // ---- kernels: one per batch bucket; ring depth from the shared memory left over
  int max_optin = 0;
  cudaDeviceGetAttribute(&max_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, e->device);
  for (int i = 0; i < 4; ++i) {
    const int bm = kBmChoices[i];
    KernelFn k = kernel_for(bm, e->hd, e->group);
    if (!k) return bail(DEC_ERR_UNSUPPORTED);
    int ring = 16;
    while (ring >= 3 && smem_layout(ring, bm, p.xmax, e->hd, e->group).total > max_optin) --ring;
    if (ring < 3) return bail(fail(e, DEC_ERR_UNSUPPORTED, "shared memory too small for the ring"));
    const int smem = smem_layout(ring, bm, p.xmax, e->hd, e->group).total;
    ce = cudaFuncSetAttribute((const void*)k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (ce != cudaSuccess) return bail(cuda_fail(e, ce, "cudaFuncSetAttribute"));
    int nb = 0;
    ce = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, (const void*)k, kThreads, smem);
    if (ce != cudaSuccess) return bail(cuda_fail(e, ce, "occupancy"));
    if (nb < 1) return bail(fail(e, DEC_ERR_UNSUPPORTED, "persistent CTA does not fit on an SM"));
    e->kern[i] = k;
    e->smem[i] = smem;
    e->ring[i] = ring;
  }
  {
    const char* tm = getenv("DEC_TIMEOUT_MS");
    double ms = tm ? atof(tm) : 1000.0;
    if (!(ms > 0)) ms = 1000.0;
    p.timeout_ns = (unsigned long long)(ms * 1e6);
    // tests only: the first q/k/v tile's layer-0 arrival is withheld, so the waits for it run out
    const char* sk = getenv("DEC_TEST_SKIP_ARRIVAL");
    p.test_skip = (sk && atoi(sk) == 1) ? 1 : 0;
    if (const char* fl = getenv("DEC_INFLIGHT")) {
      const int v = atoi(fl);
      if (v >= 1 && v <= kMaxRing) e->inflight = v;
    }
    if (const char* wm = getenv("DEC_WIDE_MIN_BATCH")) {
      const int v = atoi(wm);
      if (v >= 2 && v <= kMaxBatch + 1) e->wide_min = v;
    }
  }
  // ---- the wide kernels: steps of more than kMaxBatch tokens (own partial sums with a token
  // stride of max_batch, B operand blocks, exchange buffers)
  if (c.max_batch >= e->wide_min) {
    // the wide kernel's shape limits; an engine of at most 8 sequences that exceeds them keeps
    // every decode step on decode_step_kernel
    const int umax_w = dense ? 0 : std::min(c.n_experts, c.max_batch * c.top_k);
    const char* why = nullptr;
    {
      const long long t_max = std::max((long long)(umax_w + p.nsh) * p.n_rb_d * p.kb_i,
                                       (long long)std::max(1, umax_w) * p.n_rb_gu * p.kb_d);
      if ((t_max + 1) * G >= (1LL << 31)) why = "too many tiles in one stage";
      // the work-weighted split's positions (tiles x weight <= 8) times the grid stay 32-bit
      if ((t_max * 8 + 1) * G >= (1LL << 32)) why = "expert stage too large";
      if (!dense && c.top_k > wide::kWideTopkHost) why = "more than 8 experts per token";
      // the exponents a CTA's expert tiles read (the expert slots its range spans) fit its table
      for (int U = 0; U <= umax_w && !why; ++U)
        for (int st = 0; st < 2; ++st) {
          const int kbs = st ? p.kb_d : p.kb_i, tpe = (st ? p.n_rb_gu : p.n_rb_d) * kbs;
          const int T = (st ? U : U + p.nsh) * tpe;
          for (int cta = 0; cta < G; ++cta) {
            const int t0 = range_lo_h(T, cta, G), t1 = range_lo_h(T, cta + 1, G);
            if (t1 > t0 && ((t1 - 1) / tpe - t0 / tpe + 1) * kbs > kMaxKb) why = "expert stage too narrow";
          }
        }
    }
    if (why && c.max_batch > kMaxBatch)
      return bail(fail(e, DEC_ERR_UNSUPPORTED, std::string("decode batches above 8: ") + why));
    if (why) e->wide_min = kMaxBatch + 1;
  }
  if (c.max_batch >= e->wide_min) {
    KParams& w = e->wbase;
    w = p;
    w.MB = c.max_batch;
    const int umax_w = dense ? 0 : std::min(c.n_experts, c.max_batch * c.top_k);
    w.umax = umax_w;
    WideParams& wp = e->wp;
    wp.hmax = umax_w + p.nsh;
    const int nr_max = c.max_batch <= 16 ? 32 : c.max_batch <= 32 ? 64 : 128;
    auto wz = [&](auto** ptr, size_t bytes) -> dec_status {
      dec_status s2 = dalloc(e, ptr, bytes, &e->ws_bytes);
      if (s2 == DEC_OK && cudaMemsetAsync(*ptr, 0, bytes ? bytes : 16, e->stream) != cudaSuccess) s2 = DEC_ERR_CUDA;
      return s2;
    };
#define WZ(ptr, bytes) \
  if ((st = wz(&(ptr), (bytes))) != DEC_OK) return bail(st);
    const size_t PBS = (size_t)nr_max * 128;
    const size_t nbx = p.kb_d, nbo = p.kb_o, nbh = (size_t)wp.hmax * p.kb_i;
    const size_t nbg = (size_t)std::max(1, umax_w) * p.kb_d;
    const size_t nb = nbx + nbo + nbh + nbg;
    uint8_t* pb = nullptr;
    WZ(pb, nb * PBS);
    wp.pb = pb;
    wp.pb_bytes = nb * PBS;
    wp.pbx = pb;
    wp.pbo = pb + nbx * PBS;
    wp.pbh = pb + (nbx + nbo) * PBS;
    wp.pbg = pb + (nbx + nbo + nbh) * PBS;
    int8_t* ex = nullptr;
    WZ(ex, nb * kWideMax);
    wp.exx = ex;
    wp.exo = ex + nbx * kWideMax;
    wp.exh = ex + (nbx + nbo) * kWideMax;
    wp.exg = ex + (nbx + nbo + nbh) * kWideMax;
    WZ(wp.sel, sizeof(int32_t) * kWideMax * std::max(1, c.top_k));
    WZ(wp.selg, sizeof(float) * kWideMax * std::max(1, c.top_k));
    WZ(wp.bar, sizeof(unsigned) * 32);
    e->wnch_max = std::max(1, G / ((kMaxBatch + 1) * c.n_kv_heads));
    WZ(wp.attn_part, sizeof(float) * (size_t)w.MB * c.n_kv_heads * e->wnch_max * e->group * (c.head_dim + 2));
    WZ(wp.xbuf, (size_t)w.MB * c.hidden * 2);
    WZ(wp.xmid, (size_t)w.MB * c.hidden * 2);
    if ((st = encode_kv_map(e, &wp.kmap, p.kc, c)) != DEC_OK) return bail(st);
    if ((st = encode_kv_map(e, &wp.vmap, p.vc, c)) != DEC_OK) return bail(st);
    // partial sums: [segment][slot][MB][128] fp32 (routed stages: the largest over the expert count)
    const size_t fb = sizeof(float) * (size_t)w.MB * kTileRows;
    auto plain = [&](int kind, int n_rb) {
      return (size_t)std::max(1, n_rb) * wide::stage_slots(w, kind, 0, G);
    };
    size_t n_rtgu = 1, n_d = 1;
    for (int U = 1; U <= std::max(1, umax_w); ++U)
      n_rtgu = std::max(n_rtgu, (size_t)U * p.n_rb_gu * wide::stage_slots(w, K_RTGU, U, G));
    for (int U = 0; U <= umax_w; ++U)
      n_d = std::max(n_d, (size_t)(U + p.nsh) * p.n_rb_d * wide::stage_slots(w, K_D, U, G));
    WZ(w.part_qkv, fb * plain(K_QKV, p.n_rb_qkv));
    WZ(w.part_o, fb * plain(K_O, p.n_rb_d));
    WZ(w.part_router, fb * plain(K_ROUTER, p.n_rb_router));
    WZ(w.part_shgu, fb * plain(K_SHGU, p.n_rb_gu));
    WZ(w.part_rtgu, fb * n_rtgu);
    WZ(w.part_d, fb * n_d);
    WZ(w.part_lm, fb * plain(K_LM, p.n_rb_lm));
#undef WZ
    for (int i = 0; i < 3; ++i) {
      const int nr = 32 << i;
      if (nr > nr_max) break;
      wide::WideKernelFn k = wide::kernel_for(nr, e->hd, e->group);
      if (!k) return bail(DEC_ERR_UNSUPPORTED);
      int ring = kMaxRing;
      while (ring >= 2 && wide::smem_bytes(ring, nr, e->hd, e->group) > max_optin) --ring;
      if (ring < 2) return bail(fail(e, DEC_ERR_UNSUPPORTED, "shared memory too small for the wide ring"));
      const int smem = wide::smem_bytes(ring, nr, e->hd, e->group);
      ce = cudaFuncSetAttribute((const void*)k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      if (ce != cudaSuccess) return bail(cuda_fail(e, ce, "cudaFuncSetAttribute"));
      int nb = 0;
      ce = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, (const void*)k, kThreads, smem);
      if (ce != cudaSuccess) return bail(cuda_fail(e, ce, "occupancy"));
      if (nb < 1) return bail(fail(e, DEC_ERR_UNSUPPORTED, "wide CTA does not fit on an SM"));
      e->wkern[i] = k;
      e->wsmem[i] = smem;
      e->wring[i] = ring;
    }
    if (const char* wf = getenv("DEC_WIDE_INFLIGHT")) {
      const int v = atoi(wf);
      if (v >= 1 && v <= kMaxRing) e->winflight = v;
    }
  }
  e->lengths.assign(c.max_batch, 0);
  ce = cudaStreamSynchronize(e->stream);
  if (ce != cudaSuccess) return bail(cuda_fail(e, ce, "init synchronize"));
  *out = e;
  return DEC_OK;
}

}  // extern "C"

namespace {

// One launch of the wide kernel: B (up to 64) tokens, one per slot seq0 .. seq0 + B - 1.
dec_status launch_wide(dec_engine* e, int B, int seq0, const int32_t* tokens, const void* hidden_in, float* logits,
                       int32_t* next_tokens, void* hidden_out, cudaStream_t s) {
  const dec_model_cfg& c = e->cfg;
  const int wi = B <= 16 ? 0 : B <= 32 ? 1 : 2;
  if (B > kWideMax || !e->wkern[wi]) return fail(e, DEC_ERR_UNSUPPORTED, "no wide kernel for this batch");
  KParams p = e->wbase;
  p.B = B;
  p.seq0 = seq0;
  p.mpos = 0;
  p.accepted = nullptr;
  p.tokens = tokens;
  p.hidden_in = static_cast<const uint16_t*>(hidden_in);
  p.logits = logits;
  p.next_tokens = next_tokens;
  p.hidden_out = static_cast<uint16_t*>(hidden_out);
  p.nsteps = 1;
  p.ring = e->wring[wi];
  p.inflight = std::min(p.ring, e->winflight);
  WideParams wp = e->wp;
  wp.nch = std::max(1, std::min(e->wnch_max, e->grid / (B * c.n_kv_heads)));
  if (dec_status os = order_on(e, s)) return os;
  cudaError_t ce = cudaMemsetAsync(wp.bar, 0, sizeof(unsigned), s);
  if (ce != cudaSuccess) return cuda_fail(e, ce, "grid barrier reset");
  void* args[] = {&p, &wp};
  ce = cudaLaunchCooperativeKernel((const void*)e->wkern[wi], dim3(e->grid), dim3(kThreads), args,
                                   (size_t)e->wsmem[wi], s);
  if (ce != cudaSuccess) return cuda_fail(e, ce, "cudaLaunchCooperativeKernel (wide)");
  for (int b = 0; b < B; ++b) e->lengths[seq0 + b] += 1;
  e->launches += 1;
  return DEC_OK;
}

// One launch of the decode kernel: B tokens, either one per slot seq0 .. seq0 + B - 1, or (mpos)
// consecutive positions of slot seq0; `accepted` (device) makes it a verify step. Arguments are
// checked by the callers.
dec_status launch_step(dec_engine* e, int B, int seq0, bool mpos, const int32_t* tokens, const void* hidden_in,
                       float* logits, int32_t* next_tokens, void* hidden_out, int32_t* accepted, cudaStream_t s,
                       int nsteps = 1) {
  const dec_model_cfg& c = e->cfg;
  if (B >= e->wide_min && !mpos) {
    // (multi-position steps hold at most DEC_MAX_STEP_TOKENS <= kMaxBatch tokens and stay on
    // decode_step_kernel; generation loops one step per launch at these batches)
    if (accepted || nsteps != 1) return fail(e, DEC_ERR_ARG, "wide steps take one decode position per slot");
    return launch_wide(e, B, seq0, tokens, hidden_in, logits, next_tokens, hidden_out, s);
  }
  if (B > kMaxBatch) return fail(e, DEC_ERR_ARG, "more tokens than one step of decode_step_kernel takes");
  int bi = 0;
  while (kBmChoices[bi] < B) ++bi;
  KParams p = e->base;
  p.B = B;
  p.seq0 = seq0;
  p.mpos = mpos ? 1 : 0;
  p.accepted = accepted;
  p.tokens = tokens;
  p.hidden_in = static_cast<const uint16_t*>(hidden_in);
  p.logits = logits;
  p.next_tokens = next_tokens;
  p.hidden_out = static_cast<uint16_t*>(hidden_out);
  p.nsteps = nsteps;
  if (dec_status os = order_on(e, s)) return os;
  if (e->epoch + (unsigned)nsteps > e->epoch_limit) {
    for (const auto& b : e->epoch_bufs) {
      cudaError_t me = cudaMemsetAsync(b.first, 0, b.second, s);
      if (me != cudaSuccess) return cuda_fail(e, me, "epoch restart");
    }
    e->epoch = 0;
  }
  p.epoch = e->epoch + 1;
  e->epoch += (unsigned)nsteps;
  p.ring = e->ring[bi];
  p.inflight = std::min(p.ring, e->inflight);
  p.nch = std::max(1, std::min(e->nch_max, e->grid / (B * c.n_kv_heads)));
  void* args[] = {&p};
  cudaError_t ce = cudaLaunchCooperativeKernel((const void*)e->kern[bi], dim3(e->grid), dim3(kThreads), args,
                                               (size_t)e->smem[bi], s);
  if (ce != cudaSuccess) return cuda_fail(e, ce, "cudaLaunchCooperativeKernel");
  if (mpos) e->lengths[seq0] += B;
  else
    for (int b = 0; b < B; ++b) e->lengths[seq0 + b] += nsteps;
  e->launches += 1;
  return DEC_OK;
}

// Token-mode prefill from step-major ids tt[t][s] (device): one slot -> chunks of up to
// DEC_MAX_STEP_TOKENS consecutive positions per launch; several slots -> one launch per position
// with the slots side by side. Queued on the engine's stream.
dec_status prefill_steps(dec_engine* e, const int32_t* tt, int n_seq, int n_tokens, int seq) {
  dec_status st = DEC_OK;
  if (n_seq == 1) {
    for (int t = 0; t < n_tokens && st == DEC_OK; t += DEC_MAX_STEP_TOKENS) {
      const int n = std::min(DEC_MAX_STEP_TOKENS, n_tokens - t);
      st = launch_step(e, n, seq, true, tt + t, nullptr, nullptr, nullptr, nullptr, nullptr, e->stream);
    }
    return st;
  }
  for (int t = 0; t < n_tokens && st == DEC_OK; ++t)
    st = launch_step(e, n_seq, seq, false, tt + (size_t)t * n_seq, nullptr, nullptr, nullptr, nullptr, nullptr,
                     e->stream);
  return st;
}

// Checks shared by the multi-position entry points.
dec_status check_positions(dec_engine* e, int32_t seq, const int32_t* tokens, int32_t n) {
  if (e->poisoned) return fail(e, DEC_ERR_POISONED, "engine poisoned");
  if (dec_status ds = check_device(e)) return ds;
  const dec_model_cfg& c = e->cfg;
  if (!tokens || n < 1 || n > DEC_MAX_STEP_TOKENS || seq < 0 || seq >= c.max_batch)
    return fail(e, DEC_ERR_ARG, "positions: tokens, 1 <= n <= DEC_MAX_STEP_TOKENS, seq in range");
  if (c.vocab == 0) return fail(e, DEC_ERR_ARG, "positions need an embedding and an LM head");
  if (e->lengths[seq] + n > c.max_ctx) return fail(e, DEC_ERR_CAPACITY, "sequence full");
  return DEC_OK;
}

}  // namespace

extern "C" {

dec_status dec_step_ex(dec_engine* e, const dec_step_args* a) {
  if (!e || !a) return DEC_ERR_ARG;
  if (e->poisoned) return fail(e, DEC_ERR_POISONED, "engine poisoned");
  if (dec_status ds = check_device(e)) return ds;
  const dec_model_cfg& c = e->cfg;
  if (a->batch == 0) return DEC_OK;
  if (a->batch < 0 || a->seq0 < 0 || a->seq0 + a->batch > c.max_batch) return fail(e, DEC_ERR_ARG, "batch/seq0 out of range");
  const bool use_tokens = a->tokens != nullptr;
  if (!use_tokens && !a->hidden_in) return fail(e, DEC_ERR_ARG, "need tokens or hidden_in");
  if (use_tokens && c.vocab == 0) return fail(e, DEC_ERR_ARG, "tokens given to a headless stack");
  if ((a->logits || a->next_tokens) && c.vocab == 0) return fail(e, DEC_ERR_ARG, "no LM head");
  if (a->hidden_in && !aligned16(a->hidden_in)) return fail(e, DEC_ERR_ARG, "hidden_in must be 16-byte aligned");
  for (int b = 0; b < a->batch; ++b)
    if (e->lengths[a->seq0 + b] + 1 > c.max_ctx) return fail(e, DEC_ERR_CAPACITY, "sequence full");
  cudaStream_t s = a->stream ? static_cast<cudaStream_t>(a->stream) : e->stream;
  return launch_step(e, a->batch, a->seq0, false, a->tokens, a->hidden_in, a->logits, a->next_tokens, a->hidden_out,
                     nullptr, s);
}

dec_status dec_step_positions(dec_engine* e, int32_t seq, const int32_t* tokens, int32_t n, float* logits,
                              int32_t* next_tokens, void* stream) {
  if (!e) return DEC_ERR_ARG;
  if (dec_status cs = check_positions(e, seq, tokens, n)) return cs;
  cudaStream_t s = stream ? static_cast<cudaStream_t>(stream) : e->stream;
  return launch_step(e, n, seq, true, tokens, nullptr, logits, next_tokens, nullptr, nullptr, s);
}

dec_status dec_verify(dec_engine* e, int32_t seq, const int32_t* tokens, int32_t n, float* logits,
                      int32_t* next_tokens, int32_t* n_accepted, void* stream) {
  if (!e || !n_accepted) return DEC_ERR_ARG;
  if (dec_status cs = check_positions(e, seq, tokens, n)) return cs;
  cudaStream_t s = stream ? static_cast<cudaStream_t>(stream) : e->stream;
  const int32_t len0 = e->lengths[seq];
  dec_status st = launch_step(e, n, seq, true, tokens, nullptr, logits, next_tokens, nullptr, e->d_accepted, s);
  if (st != DEC_OK) return st;
  int32_t acc = 0;
  DEC_CUDA(cudaMemcpyAsync(&acc, e->d_accepted, sizeof(int32_t), cudaMemcpyDeviceToHost, s));
  DEC_CUDA(cudaStreamSynchronize(s));
  if (dec_status ds = check_device_status(e)) return ds;
  if (acc < 0 || acc >= n) return fail(e, DEC_ERR_DEVICE, "verify: accepted count out of range");
  e->lengths[seq] = len0 + acc + 1;  // the kernel set the device length the same way
  *n_accepted = acc;
  return DEC_OK;
}

dec_status dec_step(dec_engine* e, const int32_t* token_ids, int32_t batch, float* logits, int32_t* next_tokens,
                    void* stream) {
  dec_step_args a{};
  a.tokens = token_ids;
  a.batch = batch;
  a.logits = logits;
  a.next_tokens = next_tokens;
  a.stream = stream;
  return dec_step_ex(e, &a);
}

dec_status dec_sync(dec_engine* e) {
  if (!e) return DEC_ERR_ARG;
  if (dec_status qs = quiesce(e)) return qs;
  if (e->poisoned) return fail(e, DEC_ERR_POISONED, e->err.empty() ? "engine poisoned" : e->err);
  return check_device_status(e);
}

dec_status dec_prefill_kv(dec_engine* e, const dec_ctx* x) {
  if (!e || !x) return DEC_ERR_ARG;
  if (e->poisoned) return fail(e, DEC_ERR_POISONED, "engine poisoned");
  const dec_model_cfg& c = e->cfg;
  if (x->n_seq < 1 || x->seq < 0 || x->seq + x->n_seq > c.max_batch || x->n_tokens < 0)
    return fail(e, DEC_ERR_ARG, "bad slot range");
  if (x->n_tokens == 0) return DEC_OK;
  if (dec_status ds = check_device(e)) return ds;
  if (dec_status os = order_on(e, e->stream)) return os;  // after earlier steps, on any stream
  if (x->k_import) {
    if (!x->v_import) return fail(e, DEC_ERR_ARG, "v_import missing");
    if (x->n_tokens > c.max_ctx) return fail(e, DEC_ERR_CAPACITY, "import longer than max_ctx");
    const size_t row = (size_t)c.head_dim * 2;
    for (int s = x->seq; s < x->seq + x->n_seq; ++s)
      for (int l = 0; l < c.n_layers; ++l)
        for (int g = 0; g < c.n_kv_heads; ++g) {
          size_t src = (((size_t)l * c.n_kv_heads + g) * x->n_tokens) * row;
          size_t dst = ((((size_t)l * c.max_batch + s) * c.n_kv_heads + g) * c.max_ctx) * row;
          DEC_CUDA(cudaMemcpyAsync(reinterpret_cast<uint8_t*>(e->base.kc) + dst,
                                   static_cast<const uint8_t*>(x->k_import) + src, x->n_tokens * row,
                                   cudaMemcpyDeviceToDevice, e->stream));
          DEC_CUDA(cudaMemcpyAsync(reinterpret_cast<uint8_t*>(e->base.vc) + dst,
                                   static_cast<const uint8_t*>(x->v_import) + src, x->n_tokens * row,
                                   cudaMemcpyDeviceToDevice, e->stream));
        }
    for (int s = x->seq; s < x->seq + x->n_seq; ++s) {
      e->lengths[s] = x->n_tokens;
      DEC_CUDA(cudaMemcpyAsync(e->base.lengths + s, &e->lengths[s], sizeof(int32_t), cudaMemcpyHostToDevice, e->stream));
    }
    DEC_CUDA(cudaStreamSynchronize(e->stream));
    return DEC_OK;
  }
  if (!x->token_ids) return fail(e, DEC_ERR_ARG, "token_ids missing");
  if (c.vocab == 0) return fail(e, DEC_ERR_ARG, "token prefill needs an embedding");
  for (int s = x->seq; s < x->seq + x->n_seq; ++s)
    if (e->lengths[s] + x->n_tokens > c.max_ctx) return fail(e, DEC_ERR_CAPACITY, "prefill exceeds max_ctx");
  int32_t* tt = nullptr;
  DEC_CUDA(cudaMalloc(&tt, sizeof(int32_t) * (size_t)x->n_seq * x->n_tokens));
  const int n = x->n_seq * x->n_tokens;
  transpose_tokens_kernel<<<(n + 255) / 256, 256, 0, e->stream>>>(x->token_ids, x->n_seq, x->n_tokens, tt);
  dec_status st = prefill_steps(e, tt, x->n_seq, x->n_tokens, x->seq);
  cudaError_t ce = cudaStreamSynchronize(e->stream);
  cudaFree(tt);
  if (st != DEC_OK) return st;
  if (ce != cudaSuccess) return cuda_fail(e, ce, "prefill synchronize");
  return check_device_status(e);
}

// Token-mode prefill with the ids staged in g_prefill_ids instead of a cudaMalloc'd buffer; for
// callers that may not allocate device memory while serving (their framework's caching allocator
// holds the free memory, or cudaFree's implicit device-wide synchronisation would stall other
// streams). Overlapping calls on one device share g_prefill_ids and race; callers serialise them.
dec_status dec_prefill_kv_noalloc(dec_engine* e, const dec_ctx* x) {
  if (!e || !x) return DEC_ERR_ARG;
  if (e->poisoned) return fail(e, DEC_ERR_POISONED, "engine poisoned");
  const dec_model_cfg& c = e->cfg;
  if (x->k_import || x->v_import)
    return fail(e, DEC_ERR_ARG, "dec_prefill_kv_noalloc takes token mode only; import mode is dec_prefill_kv");
  if (x->n_seq < 1 || x->seq < 0 || x->seq + x->n_seq > c.max_batch || x->n_tokens < 0)
    return fail(e, DEC_ERR_ARG, "bad slot range");
  if (x->n_tokens == 0) return DEC_OK;
  if ((long long)x->n_seq * x->n_tokens > DEC_NOALLOC_PREFILL_MAX_IDS) {
    char buf[200];
    snprintf(buf, sizeof buf,
             "dec_prefill_kv_noalloc: n_seq * n_tokens = %lld exceeds its static scratch of %d ids; "
             "split the prompt into several calls or use dec_prefill_kv",
             (long long)x->n_seq * x->n_tokens, (int)DEC_NOALLOC_PREFILL_MAX_IDS);
    return fail(e, DEC_ERR_ARG, buf);
  }
  if (!x->token_ids) return fail(e, DEC_ERR_ARG, "token_ids missing");
  if (c.vocab == 0) return fail(e, DEC_ERR_ARG, "token prefill needs an embedding");
  for (int s = x->seq; s < x->seq + x->n_seq; ++s)
    if (e->lengths[s] + x->n_tokens > c.max_ctx) return fail(e, DEC_ERR_CAPACITY, "prefill exceeds max_ctx");
  if (dec_status ds = check_device(e)) return ds;
  int32_t* tt = nullptr;
  dec_status st = prefill_ids_scratch(e, &tt);
  if (st != DEC_OK) return st;
  // Stream order, not a device-wide wait: the transpose that overwrites the ids runs on the
  // engine's stream after the engine's earlier work (an earlier call of this engine ended with
  // its steps synchronised; other engines on the device are the caller's to serialise).
  if (dec_status os = order_on(e, e->stream)) return os;
  const int n = x->n_seq * x->n_tokens;
  transpose_tokens_kernel<<<(n + 255) / 256, 256, 0, e->stream>>>(x->token_ids, x->n_seq, x->n_tokens, tt);
  DEC_CUDA(cudaGetLastError());
  st = prefill_steps(e, tt, x->n_seq, x->n_tokens, x->seq);
  cudaError_t ce = cudaStreamSynchronize(e->stream);
  if (st != DEC_OK) return st;
  if (ce != cudaSuccess) return cuda_fail(e, ce, "prefill synchronize");
  return check_device_status(e);
}

dec_status dec_generate_device(dec_engine* e, const int32_t* first, int32_t batch, int32_t n_steps, int32_t* out,
                               void* stream) {
  if (!e || !first || !out || batch < 1 || n_steps < 0) return DEC_ERR_ARG;
  if (e->poisoned) return fail(e, DEC_ERR_POISONED, "engine poisoned");
  if (dec_status ds = check_device(e)) return ds;
  const dec_model_cfg& c = e->cfg;
  if (c.vocab == 0) return fail(e, DEC_ERR_ARG, "generate needs an LM head");
  if (batch > c.max_batch || n_steps > c.max_ctx) return fail(e, DEC_ERR_ARG, "batch or n_steps too large");
  for (int b = 0; b < batch; ++b)
    if (e->lengths[b] + n_steps > c.max_ctx) return fail(e, DEC_ERR_CAPACITY, "sequence would pass max_ctx");
  if (n_steps == 0) return DEC_OK;
  cudaStream_t s = stream ? static_cast<cudaStream_t>(stream) : e->stream;
  if (dec_status os = order_on(e, s)) return os;  // d_hist may still be read by earlier work
  const int MB = e->rows;
  DEC_CUDA(cudaMemcpy2DAsync(e->d_hist, sizeof(int32_t) * MB, first, sizeof(int32_t) * batch, sizeof(int32_t) * batch,
                             1, cudaMemcpyDeviceToDevice, s));
  // resident steps: one launch runs up to epoch_limit steps (normally all of them); wide batches
  // one step per launch, the tokens chained through d_hist on the device
  for (int i = 0; i < n_steps;) {
    const int n = batch >= e->wide_min ? 1 : std::min<int>(n_steps - i, (int)std::max(1u, e->epoch_limit));
    dec_status st = launch_step(e, batch, 0, false, e->d_hist + (size_t)i * MB, nullptr, nullptr,
                                e->d_hist + (size_t)(i + 1) * MB, nullptr, nullptr, s, n);
    if (st != DEC_OK) return st;
    i += n;
  }
  DEC_CUDA(cudaMemcpy2DAsync(out, sizeof(int32_t) * batch, e->d_hist + MB, sizeof(int32_t) * MB,
                             sizeof(int32_t) * batch, n_steps, cudaMemcpyDeviceToDevice, s));
  return DEC_OK;
}

dec_status dec_generate(dec_engine* e, const int32_t* first, int32_t batch, int32_t n_steps, int32_t* out,
                        void* stream) {
  if (!e || !first || !out || batch < 1 || n_steps < 0) return DEC_ERR_ARG;
  if (e->poisoned) return fail(e, DEC_ERR_POISONED, "engine poisoned");
  if (dec_status ds = check_device(e)) return ds;
  const dec_model_cfg& c = e->cfg;
  if (c.vocab == 0) return fail(e, DEC_ERR_ARG, "generate needs an LM head");
  if (batch > c.max_batch || n_steps > c.max_ctx) return fail(e, DEC_ERR_ARG, "batch or n_steps too large");
  for (int b = 0; b < batch; ++b)
    if (e->lengths[b] + n_steps > c.max_ctx) return fail(e, DEC_ERR_CAPACITY, "sequence would pass max_ctx");
  cudaStream_t s = stream ? static_cast<cudaStream_t>(stream) : e->stream;
  if (dec_status os = order_on(e, s)) return os;  // d_hist may still be read by earlier steps
  const int MB = e->rows;
  DEC_CUDA(cudaMemcpyAsync(e->d_hist, first, sizeof(int32_t) * batch, cudaMemcpyHostToDevice, s));
  for (int i = 0; i < n_steps;) {
    const int n = batch >= e->wide_min ? 1 : std::min<int>(n_steps - i, (int)std::max(1u, e->epoch_limit));
    dec_status st = launch_step(e, batch, 0, false, e->d_hist + (size_t)i * MB, nullptr, nullptr,
                                e->d_hist + (size_t)(i + 1) * MB, nullptr, nullptr, s, n);
    if (st != DEC_OK) return st;
    i += n;
  }
  if (n_steps > 0)
    DEC_CUDA(cudaMemcpy2DAsync(out, sizeof(int32_t) * batch, e->d_hist + MB, sizeof(int32_t) * MB,
                               sizeof(int32_t) * batch, n_steps, cudaMemcpyDeviceToHost, s));
  DEC_CUDA(cudaStreamSynchronize(s));
  if (dec_status qs = quiesce(e)) return qs;
  return check_device_status(e);
}

dec_status dec_set_length(dec_engine* e, int32_t seq, int32_t length) {
  if (!e) return DEC_ERR_ARG;
  if (seq < 0 || seq >= e->cfg.max_batch || length < 0 || length > e->cfg.max_ctx) return fail(e, DEC_ERR_ARG, "bad length");
  if (dec_status qs = quiesce(e)) return qs;  // steps may be queued on any stream
  e->lengths[seq] = length;
  DEC_CUDA(cudaMemcpyAsync(e->base.lengths + seq, &e->lengths[seq], sizeof(int32_t), cudaMemcpyHostToDevice, e->stream));
  DEC_CUDA(cudaStreamSynchronize(e->stream));
  return DEC_OK;
}

dec_status dec_get_length(dec_engine* e, int32_t seq, int32_t* length) {
  if (!e || !length || seq < 0 || seq >= e->cfg.max_batch) return DEC_ERR_ARG;
  *length = e->lengths[seq];
  return DEC_OK;
}

dec_status dec_export_kv(dec_engine* e, int32_t seq, int32_t layer, int32_t pos0, int32_t n, void* k_out, void* v_out) {
  if (!e || !k_out || !v_out) return DEC_ERR_ARG;
  const dec_model_cfg& c = e->cfg;
  if (seq < 0 || seq >= c.max_batch || layer < 0 || layer >= c.n_layers || pos0 < 0 || n < 0 || pos0 + n > c.max_ctx)
    return fail(e, DEC_ERR_ARG, "export range");
  if (dec_status os = order_on(e, e->stream)) return os;
  const size_t row = (size_t)c.head_dim * 2;
  for (int g = 0; g < c.n_kv_heads; ++g) {
    size_t src = ((((size_t)layer * c.max_batch + seq) * c.n_kv_heads + g) * c.max_ctx + pos0) * row;
    DEC_CUDA(cudaMemcpyAsync(static_cast<uint8_t*>(k_out) + (size_t)g * n * row,
                             reinterpret_cast<const uint8_t*>(e->base.kc) + src, n * row, cudaMemcpyDeviceToDevice,
                             e->stream));
    DEC_CUDA(cudaMemcpyAsync(static_cast<uint8_t*>(v_out) + (size_t)g * n * row,
                             reinterpret_cast<const uint8_t*>(e->base.vc) + src, n * row, cudaMemcpyDeviceToDevice,
                             e->stream));
  }
  DEC_CUDA(cudaStreamSynchronize(e->stream));
  return DEC_OK;
}

dec_status dec_get_info(dec_engine* e, dec_info* o) {
  if (!e || !o) return DEC_ERR_ARG;
  o->grid = e->grid;
  o->threads = kThreads;
  o->smem_bytes = e->smem[0];
  o->ring_slots = e->ring[0];
  o->stages_per_layer = 5;
  o->weight_bytes = e->weight_bytes;
  o->kv_bytes = e->kv_bytes;
  o->workspace_bytes = e->ws_bytes;
  o->launches = e->launches;
  o->wide_min_batch = e->wide_min;
  return DEC_OK;
}

dec_status dec_get_routing(dec_engine* e, int32_t layer, int32_t* idx, float* gates) {
  if (!e || !idx || !gates) return DEC_ERR_ARG;
  const dec_model_cfg& c = e->cfg;
  if (c.n_experts == 0 || layer < 0 || layer >= c.n_layers) return fail(e, DEC_ERR_ARG, "no routing for this layer");
  if (dec_status os = order_on(e, e->stream)) return os;
  const size_t n = (size_t)e->rows * c.top_k, off = (size_t)layer * n;
  DEC_CUDA(cudaMemcpyAsync(idx, e->base.rt_idx + off, sizeof(int32_t) * n, cudaMemcpyDeviceToHost, e->stream));
  DEC_CUDA(cudaMemcpyAsync(gates, e->base.rt_topk_gate + off, sizeof(float) * n, cudaMemcpyDeviceToHost, e->stream));
  DEC_CUDA(cudaStreamSynchronize(e->stream));
  return DEC_OK;
}

dec_status dec_get_router_logits(dec_engine* e, int32_t layer, float* logits) {
  if (!e || !logits) return DEC_ERR_ARG;
  const dec_model_cfg& c = e->cfg;
  if (c.n_experts == 0 || layer < 0 || layer >= c.n_layers) return fail(e, DEC_ERR_ARG, "no routing for this layer");
  if (dec_status os = order_on(e, e->stream)) return os;
  const size_t n = (size_t)e->rows * c.n_experts;
  DEC_CUDA(cudaMemcpyAsync(logits, e->base.rt_logits + (size_t)layer * n, sizeof(float) * n, cudaMemcpyDeviceToHost,
                           e->stream));
  DEC_CUDA(cudaStreamSynchronize(e->stream));
  return DEC_OK;
}

dec_status dec_get_trace(dec_engine* e, uint64_t* host_buf, int32_t n, int32_t* n_written) {
  if (!e || !host_buf || n < 0) return DEC_ERR_ARG;
  if (dec_status os = order_on(e, e->stream)) return os;
  const int m = std::min(n, kTraceSlots + kBarTrace * e->grid);
  DEC_CUDA(cudaMemcpyAsync(host_buf, e->base.trace, sizeof(uint64_t) * m, cudaMemcpyDeviceToHost, e->stream));
  DEC_CUDA(cudaStreamSynchronize(e->stream));
  if (n_written) *n_written = m;
  return DEC_OK;
}

dec_status dec_get_layer_times(dec_engine* e, uint64_t* host_buf, int32_t n, int32_t* n_written) {
  if (!e || !host_buf || n < 0) return DEC_ERR_ARG;
  if (dec_status os = order_on(e, e->stream)) return os;
  const int m = std::min(n, e->cfg.n_layers + 2);
  DEC_CUDA(cudaMemcpyAsync(host_buf, e->base.layer_ts, sizeof(uint64_t) * m, cudaMemcpyDeviceToHost, e->stream));
  DEC_CUDA(cudaStreamSynchronize(e->stream));
  if (n_written) *n_written = m;
  return DEC_OK;
}

const char* dec_last_error(const dec_engine* e) { return e ? e->err.c_str() : "no engine"; }

void dec_destroy(dec_engine* e) {
  if (!e) return;
  if (e->stream && e->order_ev) quiesce(e);
  for (void* p : e->allocs) cudaFree(p);
  if (e->order_ev) cudaEventDestroy(e->order_ev);
  if (e->stream) cudaStreamDestroy(e->stream);
  delete e;
}

}  // extern "C"
