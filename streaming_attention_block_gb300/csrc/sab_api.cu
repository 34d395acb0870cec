// Host side of libsab.so: ring handle, argument validation, key-set planner,
// TMA tensor-map encoding and kernel launches.  No call allocates device
// memory or synchronises the host (except sab_get_last_device_error).
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <new>
#include <vector>

#include "../../include/sab.h"
#include "sab_internal.h"

using namespace sab;

namespace {

constexpr size_t kAlign = 256;

// Debug builds: the kind of launch whose next instance carries a forged index
// (sab_debug_inject_bounds_error); 0 when none is pending.
std::atomic<int> g_inject{0};
bool take_injection(int what) {
  if (!kDebugBounds) return false;
  int expect = what;
  return g_inject.compare_exchange_strong(expect, 0);
}
size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                  CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                  CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// 4-D bf16 map with coordinates (d, row, h, b) and a 64 x 128 box, 128-byte swizzle.
bool encode_map(CUtensorMap* m, const void* ptr, int D, long long rows, int H, int B, size_t s_row,
                size_t s_h, size_t s_b, int box_rows = kTileN) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)rows, (cuuint64_t)H, (cuuint64_t)B};
  const cuuint64_t strides[3] = {(cuuint64_t)s_row, (cuuint64_t)s_h, (cuuint64_t)s_b};
  const cuuint32_t box[4] = {64, (cuuint32_t)box_rows, 1, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Head-major [B, H, rows, D] E4M3 codes: plain (unswizzled) 128-row boxes of
// whole D-byte rows, expanded to bf16 inside the attention kernel.
bool encode_head_major_u8(CUtensorMap* m, const void* ptr, int B, int H, long long rows, int D,
                          bool swizzle128 = false) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)rows, (cuuint64_t)H, (cuuint64_t)B};
  const cuuint64_t strides[3] = {(cuuint64_t)D, (cuuint64_t)rows * D, (cuuint64_t)H * rows * D};
  const cuuint32_t box[4] = {(cuuint32_t)D, (cuuint32_t)kTileN, 1, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(ptr), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Token-major [B, L, H, D] bf16.
bool encode_token_major(CUtensorMap* m, const void* ptr, int B, int L, int H, int D, int box_rows = kTileN) {
  const size_t e = 2;
  return encode_map(m, ptr, D, L, H, B, (size_t)H * D * e, (size_t)D * e, (size_t)L * H * D * e, box_rows);
}

// Head-major [B, H, rows, D] bf16.
bool encode_head_major(CUtensorMap* m, const void* ptr, int B, int H, long long rows, int D) {
  const size_t e = 2;
  return encode_map(m, ptr, D, rows, H, B, (size_t)D * e, (size_t)rows * D * e, (size_t)H * rows * D * e);
}

bool valid_desc(const sab_ring_desc* d) {
  if (d == nullptr) return false;
  if (d->num_layers < 1 || d->batch < 1 || d->heads < 1 || d->chunk_tokens < 1 || d->ring_slots < 1)
    return false;
  if (d->head_dim != 64 && d->head_dim != 128) return false;
  if (d->has_sink != 0 && d->has_sink != 1) return false;
  if (d->kv_dtype != SAB_KV_BF16 && d->kv_dtype != SAB_KV_FP8_E4M3 && d->kv_dtype != SAB_KV_INT8K_FP8V)
    return false;
  const long long rows = (long long)(d->has_sink + d->ring_slots) * d->chunk_tokens;
  if (rows > (1LL << 30)) return false;
  if ((long long)d->batch * d->heads * rows * d->head_dim > (1LL << 40)) return false;
  return true;
}

struct Geometry {
  long long rows;       // rows per (b, h)
  size_t codes_bytes;   // one tensor (K or V) of one layer, aligned
  size_t scale_bytes;   // one tensor's scales of one layer, aligned (FP8)
  size_t layer_bytes;
};

Geometry geometry(const sab_ring_desc& d) {
  Geometry g;
  g.rows = (long long)(d.has_sink + d.ring_slots) * d.chunk_tokens;
  const size_t esize = d.kv_dtype == SAB_KV_BF16 ? 2 : 1;
  g.codes_bytes = align_up((size_t)d.batch * d.heads * g.rows * d.head_dim * esize, kAlign);
  g.scale_bytes = d.kv_dtype != SAB_KV_BF16
                      ? align_up((size_t)d.batch * d.heads * (d.has_sink + d.ring_slots) * sizeof(float), kAlign)
                      : 0;
  g.layer_bytes = 2 * g.codes_bytes + 2 * g.scale_bytes;
  return g;
}

// Split workspace: one arrival counter per (b, h, query tile), then the
// fp32 partial rows [S][B*H][n_qtiles*128][D] and partial LSEs [S][B*H][n_qtiles*128].
struct WsLayout {
  size_t count_off, o_off, lse_off, total;
};
WsLayout ws_layout(int BH, int Lq, int D, int splits) {
  WsLayout w{0, 0, 0, 0};
  if (splits <= 1) return w;
  const size_t n_qtiles = (size_t)(Lq + kTileM - 1) / kTileM;
  const size_t lq_pad = n_qtiles * kTileM;
  w.count_off = 0;
  w.o_off = align_up((size_t)BH * n_qtiles * sizeof(unsigned), kAlign);
  w.lse_off = w.o_off + align_up((size_t)splits * BH * lq_pad * D * sizeof(float), kAlign);
  w.total = w.lse_off + align_up((size_t)splits * BH * lq_pad * sizeof(float), kAlign);
  return w;
}

constexpr int kMaxSplits = 256;
constexpr int kMaxAutoSplits = 8;

int device_sms() {
  static int n = 0;
  if (n == 0) {
    int dev = 0, v = 0;
    if (cudaGetDevice(&dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && v > 0)
      n = v;
    else
      return 148;
  }
  return n;
}

// num_splits == 0: the KV split count S (1..8) that minimises the modelled
// time of one call, in key-tile periods.  CTAs (one query tile x one split)
// run one per SM, so the call takes ceil(tiles * S / SMs) waves of
// ceil(kv_tiles / S) key tiles each; every wave after the first also pays a
// CTA's set-up and epilogue (about 5 key tiles: the first wave's overlaps the
// previous kernel), and S > 1 adds the partial-tile write and the merge (about
// 1 + 0.4 S key tiles).
int auto_splits(long long q_tiles, int kv_tiles) {
  const long long sms = device_sms();
  int best = 1;
  double best_cost = 0.0;
  for (int s = 1; s <= kMaxAutoSplits && (s == 1 || s <= kv_tiles / 2); ++s) {
    const long long waves = (q_tiles * s + sms - 1) / sms;
    double cost = (double)waves * ((kv_tiles + s - 1) / s) + 5.0 * (double)(waves - 1);
    if (s > 1) cost += 1.0 + 0.4 * s;
    if (s == 1 || cost < best_cost) {
      best_cost = cost;
      best = s;
    }
  }
  return best;
}

}  // namespace

struct sab_ring {
  sab_ring_desc d;
  uint8_t* mem;
  Geometry g;
  std::vector<long long> newest;
  std::vector<int> held;
  std::vector<int> sink_set;
  std::vector<CUtensorMap> kmap, vmap;  // per layer, BF16 rings

  uint8_t* layer_base(int l) const { return mem + (size_t)l * g.layer_bytes; }
  void* k(int l) const { return layer_base(l); }
  void* v(int l) const { return layer_base(l) + g.codes_bytes; }
  float* ks(int l) const {
    return g.scale_bytes ? reinterpret_cast<float*>(layer_base(l) + 2 * g.codes_bytes) : nullptr;
  }
  float* vs(int l) const {
    return g.scale_bytes ? reinterpret_cast<float*>(layer_base(l) + 2 * g.codes_bytes + g.scale_bytes) : nullptr;
  }
};

extern "C" {

size_t sab_kv_ring_bytes(const sab_ring_desc* desc) {
  if (!valid_desc(desc)) return 0;
  return geometry(*desc).layer_bytes * (size_t)desc->num_layers;
}

sab_status sab_kv_ring_create(const sab_ring_desc* desc, void* dev_mem, size_t bytes, void* stream,
                              sab_ring** out) {
  if (out == nullptr || !valid_desc(desc) || dev_mem == nullptr) return SAB_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(dev_mem) % kAlign) != 0) return SAB_ERR_INVALID_ARG;
  const size_t need = sab_kv_ring_bytes(desc);
  if (bytes < need) return SAB_ERR_INVALID_ARG;
  sab_ring* r = new (std::nothrow) sab_ring();
  if (r == nullptr) return SAB_ERR_INVALID_ARG;
  r->d = *desc;
  r->mem = static_cast<uint8_t*>(dev_mem);
  r->g = geometry(*desc);
  r->newest.assign(desc->num_layers, -1);
  r->held.assign(desc->num_layers, 0);
  r->sink_set.assign(desc->num_layers, 0);
  r->kmap.resize(desc->num_layers);
  r->vmap.resize(desc->num_layers);
  const bool fp8 = desc->kv_dtype != SAB_KV_BF16;  // one byte per element
  for (int l = 0; l < desc->num_layers; ++l) {
    const int B = desc->batch, H = desc->heads, D = desc->head_dim;
    const bool okm = fp8 ? (encode_head_major_u8(&r->kmap[l], r->k(l), B, H, r->g.rows, D) &&
                            encode_head_major_u8(&r->vmap[l], r->v(l), B, H, r->g.rows, D))
                         : (encode_head_major(&r->kmap[l], r->k(l), B, H, r->g.rows, D) &&
                            encode_head_major(&r->vmap[l], r->v(l), B, H, r->g.rows, D));
    if (!okm) {
      delete r;
      return SAB_ERR_CUDA;
    }
  }
  if (cudaMemsetAsync(dev_mem, 0, need, static_cast<cudaStream_t>(stream)) != cudaSuccess) {
    delete r;
    return SAB_ERR_CUDA;
  }
  *out = r;
  return SAB_OK;
}

sab_status sab_kv_ring_destroy(sab_ring* ring) {
  delete ring;
  return SAB_OK;
}

sab_status sab_kv_ring_get_desc(const sab_ring* ring, sab_ring_desc* desc) {
  if (ring == nullptr || desc == nullptr) return SAB_ERR_INVALID_ARG;
  *desc = ring->d;
  return SAB_OK;
}

sab_status sab_kv_ring_layer_ptrs(const sab_ring* ring, int layer, void** k, void** v, float** k_scale,
                                  float** v_scale) {
  if (ring == nullptr || layer < 0 || layer >= ring->d.num_layers) return SAB_ERR_INVALID_ARG;
  if (k) *k = ring->k(layer);
  if (v) *v = ring->v(layer);
  if (k_scale) *k_scale = ring->ks(layer);
  if (v_scale) *v_scale = ring->vs(layer);
  return SAB_OK;
}

static sab_status write_chunk(sab_ring* r, int layer, int slot_row0, int scale_idx, const void* K, const void* V,
                              void* stream, const long long* d_chunk = nullptr) {
  AppendParams p;
  memset(&p, 0, sizeof(p));
  p.src[0] = static_cast<const uint16_t*>(K);
  p.src[1] = static_cast<const uint16_t*>(V);
  p.dst[0] = r->k(layer);
  p.dst[1] = r->v(layer);
  p.scale[0] = r->ks(layer);
  p.scale[1] = r->vs(layer);
  p.B = r->d.batch;
  p.H = r->d.heads;
  p.D = r->d.head_dim;
  p.Lc = r->d.chunk_tokens;
  p.rows = (int)r->g.rows;
  p.slot_row0 = slot_row0;
  p.scale_idx = scale_idx;
  p.scale_stride = r->d.has_sink + r->d.ring_slots;
  p.k_int8 = r->d.kv_dtype == SAB_KV_INT8K_FP8V ? 1 : 0;
  p.d_chunk = d_chunk;
  p.ring_slots = r->d.ring_slots;
  p.has_sink = r->d.has_sink;
  p.err_word = device_error_word();
  if (d_chunk == nullptr && take_injection(SAB_DEBUG_INJECT_APPEND_SLOT)) {
    p.slot_row0 = p.rows;  // one slot past the (b, h) block
    p.scale_idx = p.scale_stride;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const cudaError_t e = r->d.kv_dtype == SAB_KV_BF16 ? launch_append_bf16(p, s) : launch_append_fp8(p, s);
  return e == cudaSuccess ? SAB_OK : SAB_ERR_CUDA;
}

sab_status sab_kv_ring_set_sink(sab_ring* ring, int layer, const void* K, const void* V, void* stream) {
  if (ring == nullptr || layer < 0 || layer >= ring->d.num_layers) return SAB_ERR_INVALID_ARG;
  if (K == nullptr || V == nullptr || !aligned16(K) || !aligned16(V)) return SAB_ERR_INVALID_ARG;
  if (!ring->d.has_sink) return SAB_ERR_UNSUPPORTED;
  const sab_status st = write_chunk(ring, layer, 0, 0, K, V, stream);
  if (st == SAB_OK) ring->sink_set[layer] = 1;
  return st;
}

sab_status sab_kv_ring_append(sab_ring* ring, int layer, long long chunk, const void* K, const void* V,
                              void* stream) {
  if (ring == nullptr || layer < 0 || layer >= ring->d.num_layers) return SAB_ERR_INVALID_ARG;
  if (K == nullptr || V == nullptr || !aligned16(K) || !aligned16(V)) return SAB_ERR_INVALID_ARG;
  if (chunk < 0) return SAB_ERR_OUT_OF_RANGE;
  const long long newest = ring->newest[layer];
  if (newest >= 0 && chunk != newest && chunk != newest + 1) return SAB_ERR_OUT_OF_RANGE;
  const int R = ring->d.ring_slots;
  const int slot = (int)(chunk % R);
  const int row0 = (ring->d.has_sink + slot) * ring->d.chunk_tokens;
  const sab_status st = write_chunk(ring, layer, row0, ring->d.has_sink + slot, K, V, stream);
  if (st != SAB_OK) return st;
  if (newest < 0) {
    ring->held[layer] = 1;
  } else if (chunk == newest + 1) {
    ring->held[layer] = std::min(R, ring->held[layer] + 1);
  }
  ring->newest[layer] = chunk;
  return SAB_OK;
}

sab_status sab_kv_ring_slot_of(const sab_ring* ring, int layer, long long chunk, int* slot) {
  if (ring == nullptr || slot == nullptr || layer < 0 || layer >= ring->d.num_layers) return SAB_ERR_INVALID_ARG;
  const long long newest = ring->newest[layer];
  if (newest < 0 || chunk > newest || chunk <= newest - ring->held[layer]) return SAB_ERR_OUT_OF_RANGE;
  *slot = (int)(chunk % ring->d.ring_slots);
  return SAB_OK;
}

sab_status sab_kv_ring_get_state(const sab_ring* ring, long long* newest_chunk, int* held, int* sink_set) {
  if (ring == nullptr) return SAB_ERR_INVALID_ARG;
  for (int l = 0; l < ring->d.num_layers; ++l) {
    if (newest_chunk) newest_chunk[l] = ring->newest[l];
    if (held) held[l] = ring->held[l];
    if (sink_set) sink_set[l] = ring->sink_set[l];
  }
  return SAB_OK;
}

sab_status sab_kv_ring_set_state(sab_ring* ring, const long long* newest_chunk, const int* held,
                                 const int* sink_set) {
  if (ring == nullptr || newest_chunk == nullptr || held == nullptr || sink_set == nullptr)
    return SAB_ERR_INVALID_ARG;
  for (int l = 0; l < ring->d.num_layers; ++l) {
    const long long n = newest_chunk[l];
    const int h = held[l];
    if (n < -1 || h < 0 || h > ring->d.ring_slots || (long long)h > n + 1 || ((n == -1) != (h == 0)))
      return SAB_ERR_INVALID_ARG;
    if (sink_set[l] != 0 && sink_set[l] != 1) return SAB_ERR_INVALID_ARG;
    if (sink_set[l] && !ring->d.has_sink) return SAB_ERR_INVALID_ARG;
  }
  for (int l = 0; l < ring->d.num_layers; ++l) {
    ring->newest[l] = newest_chunk[l];
    ring->held[l] = held[l];
    ring->sink_set[l] = sink_set[l];
  }
  return SAB_OK;
}

size_t sab_chunk_attention_workspace(const sab_ring* ring, int num_splits) {
  if (ring == nullptr || num_splits < 0 || num_splits > kMaxSplits) return 0;
  if (num_splits == 0) num_splits = kMaxAutoSplits;
  return ws_layout(ring->d.batch * ring->d.heads, ring->d.chunk_tokens, ring->d.head_dim, num_splits).total;
}

static sab_status launch_attention(AttnParams& p, int Lq, int splits, void* workspace, size_t ws_bytes,
                                   void* stream) {
  if ((long long)p.B * p.H > 65535) return SAB_ERR_UNSUPPORTED;
  // One CTA per (128-query tile, (b, h), KV split), key-half softmax.  Splits
  // (explicit, or chosen on auto to fill the SMs) merge their partial rows by
  // log-sum-exp through the workspace.
  const int n_qtiles = (Lq + kTileM - 1) / kTileM;
  if (splits == 0) {
    // block-causal: a query tile sees at most (window + 1) chunks plus one straddled tile
    const int tiles = p.mode == kModeStreaming
                          ? p.plan.total_tiles
                          : ((p.window + 1) * p.chunk_tokens + 2 * kTileN - 1) / kTileN;
    splits = auto_splits((long long)n_qtiles * p.B * p.H, tiles);
  }
  p.Lq = Lq;
  p.n_qtiles = n_qtiles;
  p.splits = splits;
  if (splits > 1) {
    const WsLayout w = ws_layout(p.B * p.H, Lq, p.D, splits);
    if (workspace == nullptr || ws_bytes < w.total) return SAB_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) % kAlign) != 0) return SAB_ERR_INVALID_ARG;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    p.ws_count = reinterpret_cast<unsigned*>(ws + w.count_off);
    p.ws_o = reinterpret_cast<float*>(ws + w.o_off);
    p.ws_lse = reinterpret_cast<float*>(ws + w.lse_off);
    p.ws_tiles = (long long)((w.lse_off - w.o_off) / ((size_t)kTileM * p.D * sizeof(float)));
    if (take_injection(SAB_DEBUG_INJECT_WS_TILE)) p.ws_tiles -= 1;  // the last tile "past" the workspace
  }
  if (p.mode == kModeStreaming && p.d_chunk == nullptr && p.plan.nseg > 0 &&
      take_injection(SAB_DEBUG_INJECT_KEY_ROW)) {
    KvSegment& sg = p.plan.seg[p.plan.nseg - 1];
    sg.row0 += p.src_rows[sg.src];  // the last key run moved past the end of its source
  }
  return launch_chunk_attention_kh(p, static_cast<cudaStream_t>(stream)) == cudaSuccess ? SAB_OK : SAB_ERR_CUDA;
}

// Validation and key-set planning shared by both chunk-attention entry points.
// Validation and parameters common to host-planned and graph-mode calls
// (everything but the chunk index).
static sab_status plan_common(const sab_ring* ring, int layer, const void* Q, const void* K_cur, const void* V_cur,
                              int window, int use_sink, int num_splits, float softmax_scale, void* O, float* LSE,
                              AttnParams& p) {
  if (ring == nullptr || layer < 0 || layer >= ring->d.num_layers) return SAB_ERR_INVALID_ARG;
  if (Q == nullptr || O == nullptr || !aligned16(Q) || !aligned16(O)) return SAB_ERR_INVALID_ARG;
  if ((K_cur == nullptr) != (V_cur == nullptr)) return SAB_ERR_INVALID_ARG;
  if (K_cur != nullptr && (!aligned16(K_cur) || !aligned16(V_cur))) return SAB_ERR_INVALID_ARG;
  if (LSE != nullptr && (reinterpret_cast<uintptr_t>(LSE) & 3u) != 0) return SAB_ERR_INVALID_ARG;
  if (window < 0 || num_splits < 0 || num_splits > kMaxSplits) return SAB_ERR_INVALID_ARG;
  if (!(softmax_scale > 0.f) || !isfinite(softmax_scale)) return SAB_ERR_INVALID_ARG;
  if (use_sink != 0 && use_sink != 1) return SAB_ERR_INVALID_ARG;
  const sab_ring_desc& d = ring->d;
  if (use_sink && !d.has_sink) return SAB_ERR_INVALID_ARG;
  if (use_sink && !ring->sink_set[layer]) return SAB_ERR_OUT_OF_RANGE;
  const bool kcur = K_cur != nullptr;
  const bool fp8 = d.kv_dtype != SAB_KV_BF16;
  // The 8-bit cache path expands 128-byte code rows in place (D = 128), reads
  // every key from the ring (the current chunk is appended first) and needs
  // chunks of at least 128 tokens (a key tile spans at most two chunks).
  if (fp8 && (kcur || d.head_dim != 128 || d.chunk_tokens < kTileN)) return SAB_ERR_UNSUPPORTED;
  const int Lc = d.chunk_tokens;
  memset(&p, 0, sizeof(p));
  p.mode = kModeStreaming;
  p.fp8 = fp8 ? 1 : 0;
  p.k_int8 = d.kv_dtype == SAB_KV_INT8K_FP8V ? 1 : 0;
  p.k_scale = ring->ks(layer);
  p.v_scale = ring->vs(layer);
  p.scale_stride = d.has_sink + d.ring_slots;
  p.chunk_tokens = d.chunk_tokens;
  p.B = d.batch;
  p.H = d.heads;
  p.D = d.head_dim;
  p.scale_log2 = softmax_scale * 1.4426950408889634f;
  p.O = static_cast<uint16_t*>(O);
  p.LSE = LSE;
  p.window = window;
  p.ring_slots = d.ring_slots;
  p.has_sink = d.has_sink;
  p.use_sink = use_sink;
  p.kcur = kcur ? 1 : 0;
  p.src_rows[0] = (int)ring->g.rows;
  p.src_rows[1] = kcur ? Lc : 0;
  p.k_map[0] = ring->kmap[layer];
  p.v_map[0] = ring->vmap[layer];
  p.k_map[1] = ring->kmap[layer];
  p.v_map[1] = ring->vmap[layer];
  if (kcur) {
    if (!encode_token_major(&p.k_map[1], K_cur, d.batch, Lc, d.heads, d.head_dim) ||
        !encode_token_major(&p.v_map[1], V_cur, d.batch, Lc, d.heads, d.head_dim))
      return SAB_ERR_CUDA;
  }
  if (!encode_token_major(&p.q_map, Q, d.batch, Lc, d.heads, d.head_dim) ||
      !encode_token_major(&p.o_map, O, d.batch, Lc, d.heads, d.head_dim))
    return SAB_ERR_CUDA;
  return SAB_OK;
}

// Validation and key-set planning of a host-planned call (chunk known here).
static sab_status plan_chunk_attention(const sab_ring* ring, int layer, long long chunk, const void* Q,
                                       const void* K_cur, const void* V_cur, int window, int use_sink,
                                       int num_splits, float softmax_scale, void* O, float* LSE, AttnParams& p) {
  const sab_status st =
      plan_common(ring, layer, Q, K_cur, V_cur, window, use_sink, num_splits, softmax_scale, O, LSE, p);
  if (st != SAB_OK) return st;
  if (chunk < 0) return SAB_ERR_OUT_OF_RANGE;
  // ring chunks needed: [need_lo, need_hi], all held by the ring
  const long long need_lo = std::max(0LL, chunk - window);
  const long long need_hi = p.kcur ? chunk - 1 : chunk;
  if (need_hi >= need_lo) {
    const long long newest = ring->newest[layer];
    const long long oldest = newest - ring->held[layer] + 1;
    if (newest < 0 || need_hi > newest || need_lo < oldest) return SAB_ERR_OUT_OF_RANGE;
  }
  plan_key_runs(chunk, window, p.ring_slots, p.chunk_tokens, p.has_sink, use_sink, p.kcur, p.plan);
  return SAB_OK;
}

sab_status sab_chunk_attention(const sab_ring* ring, int layer, long long chunk, const void* Q, const void* K_cur,
                               const void* V_cur, int window, int use_sink, int num_splits, float softmax_scale,
                               void* O, float* LSE, void* workspace, size_t ws_bytes, void* stream) {
  AttnParams p;
  const sab_status st =
      plan_chunk_attention(ring, layer, chunk, Q, K_cur, V_cur, window, use_sink, num_splits, softmax_scale, O, LSE, p);
  if (st != SAB_OK) return st;
  return launch_attention(p, ring->d.chunk_tokens, num_splits, workspace, ws_bytes, stream);
}

sab_status sab_chunk_attention_fp8mma(const sab_ring* ring, int layer, long long chunk, const void* Q, int window,
                                      int use_sink, int num_splits, float softmax_scale, void* O, float* LSE,
                                      void* workspace, size_t ws_bytes, void* stream) {
  if (ring == nullptr) return SAB_ERR_INVALID_ARG;
  if (ring->d.kv_dtype != SAB_KV_FP8_E4M3) return SAB_ERR_UNSUPPORTED;
  AttnParams p;
  const sab_status st = plan_chunk_attention(ring, layer, chunk, Q, nullptr, nullptr, window, use_sink, num_splits,
                                             softmax_scale, O, LSE, p);
  if (st != SAB_OK) return st;
  p.f8mma = 1;
  // the tensor cores read the code tiles as K-major / MN-major operands in
  // the 128-byte-swizzled layout (D = 128 codes = one swizzle row)
  const sab_ring_desc& d = ring->d;
  if (!encode_head_major_u8(&p.k_map[0], ring->k(layer), d.batch, d.heads, ring->g.rows, d.head_dim, true) ||
      !encode_head_major_u8(&p.v_map[0], ring->v(layer), d.batch, d.heads, ring->g.rows, d.head_dim, true))
    return SAB_ERR_CUDA;
  return launch_attention(p, ring->d.chunk_tokens, num_splits, workspace, ws_bytes, stream);
}

sab_status sab_chunk_attention_dev(const sab_ring* ring, int layer, const long long* d_chunk, const void* Q,
                                   const void* K_cur, const void* V_cur, int window, int use_sink, int num_splits,
                                   float softmax_scale, void* O, float* LSE, void* workspace, size_t ws_bytes,
                                   void* stream) {
  if (d_chunk == nullptr || (reinterpret_cast<uintptr_t>(d_chunk) & 7u) != 0) return SAB_ERR_INVALID_ARG;
  AttnParams p;
  const sab_status st =
      plan_common(ring, layer, Q, K_cur, V_cur, window, use_sink, num_splits, softmax_scale, O, LSE, p);
  if (st != SAB_OK) return st;
  // every window the stream can ask for must fit in the ring
  if (window > (p.kcur ? p.ring_slots : p.ring_slots - 1)) return SAB_ERR_OUT_OF_RANGE;
  p.d_chunk = d_chunk;
  // the host plan of a full window sizes the split choice; the kernels plan
  // the actual chunk on the device
  plan_key_runs((long long)window + p.ring_slots, window, p.ring_slots, p.chunk_tokens, p.has_sink, use_sink,
                p.kcur, p.plan);
  return launch_attention(p, ring->d.chunk_tokens, num_splits, workspace, ws_bytes, stream);
}

sab_status sab_qk_norm_rope(sab_ring* ring, int layer, long long chunk, const void* Q, const void* K, const void* V,
                            const float* gamma_q, const float* gamma_k, const sab_rope_desc* rope, void* Q_out,
                            void* K_out, void* V_out, int append, void* stream) {
  if (ring == nullptr || layer < 0 || layer >= ring->d.num_layers || rope == nullptr) return SAB_ERR_INVALID_ARG;
  const sab_ring_desc& d = ring->d;
  if (Q == nullptr || K == nullptr || V == nullptr || Q_out == nullptr) return SAB_ERR_INVALID_ARG;
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(Q_out)) return SAB_ERR_INVALID_ARG;
  if ((K_out && !aligned16(K_out)) || (V_out && !aligned16(V_out))) return SAB_ERR_INVALID_ARG;
  if ((gamma_q && (reinterpret_cast<uintptr_t>(gamma_q) & 3u)) || (gamma_k && (reinterpret_cast<uintptr_t>(gamma_k) & 3u)))
    return SAB_ERR_INVALID_ARG;
  if (append != 0 && append != 1) return SAB_ERR_INVALID_ARG;
  if (rope->frames < 1 || rope->height < 1 || rope->width < 1 ||
      (long long)rope->frames * rope->height * rope->width != d.chunk_tokens)
    return SAB_ERR_INVALID_ARG;
  if (rope->band_t < 0 || rope->band_h < 0 || rope->band_w < 0 || (rope->band_t | rope->band_h | rope->band_w) & 1 ||
      rope->band_t + rope->band_h + rope->band_w != d.head_dim)
    return SAB_ERR_INVALID_ARG;
  if (!(rope->base > 1.f) || !isfinite(rope->base) || !(rope->eps > 0.f) || !isfinite(rope->eps))
    return SAB_ERR_INVALID_ARG;
  if (chunk < 0) return SAB_ERR_OUT_OF_RANGE;
  const bool bf16_ring = d.kv_dtype == SAB_KV_BF16;
  // an 8-bit ring quantises per (batch, head) block: K', V go through K_out,
  // V_out and the ring's own quantiser
  if (append && !bf16_ring && (K_out == nullptr || V_out == nullptr)) return SAB_ERR_INVALID_ARG;
  const long long newest = ring->newest[layer];
  if (append && newest >= 0 && chunk != newest && chunk != newest + 1) return SAB_ERR_OUT_OF_RANGE;
  const int R = d.ring_slots, slot = (int)(chunk % R);
  RopeParams rp;
  memset(&rp, 0, sizeof(rp));
  rp.q_in = static_cast<const uint16_t*>(Q);
  rp.k_in = static_cast<const uint16_t*>(K);
  rp.v_in = static_cast<const uint16_t*>(V);
  rp.gamma_q = gamma_q;
  rp.gamma_k = gamma_k;
  rp.q_out = static_cast<uint16_t*>(Q_out);
  rp.k_out = static_cast<uint16_t*>(K_out);
  rp.v_out = static_cast<uint16_t*>(V_out);
  if (append && bf16_ring) {
    rp.ring_k = static_cast<uint16_t*>(ring->k(layer));
    rp.ring_v = static_cast<uint16_t*>(ring->v(layer));
  }
  rp.B = d.batch;
  rp.H = d.heads;
  rp.D = d.head_dim;
  rp.Lc = d.chunk_tokens;
  rp.rows = (int)ring->g.rows;
  rp.slot_row0 = (d.has_sink + slot) * d.chunk_tokens;
  rp.err_word = device_error_word();
  if (rp.ring_k != nullptr && take_injection(SAB_DEBUG_INJECT_APPEND_SLOT)) rp.slot_row0 = rp.rows;
  rp.chunk = chunk;
  rp.F = rope->frames;
  rp.Hp = rope->height;
  rp.Wp = rope->width;
  rp.bt = rope->band_t;
  rp.bh = rope->band_h;
  rp.bw = rope->band_w;
  rp.log2_base = log2f(rope->base);
  rp.eps = rope->eps;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (launch_qk_rope(rp, s) != cudaSuccess) return SAB_ERR_CUDA;
  if (!append) return SAB_OK;
  if (!bf16_ring) {
    const sab_status st = write_chunk(ring, layer, rp.slot_row0, d.has_sink + slot, K_out, V_out, stream);
    if (st != SAB_OK) return st;
  }
  if (newest < 0) {
    ring->held[layer] = 1;
  } else if (chunk == newest + 1) {
    ring->held[layer] = std::min(R, ring->held[layer] + 1);
  }
  ring->newest[layer] = chunk;
  return SAB_OK;
}

sab_status sab_kv_ring_append_dev(sab_ring* ring, int layer, const long long* d_chunk, const void* K,
                                  const void* V, void* stream) {
  if (ring == nullptr || layer < 0 || layer >= ring->d.num_layers) return SAB_ERR_INVALID_ARG;
  if (K == nullptr || V == nullptr || !aligned16(K) || !aligned16(V)) return SAB_ERR_INVALID_ARG;
  if (d_chunk == nullptr || (reinterpret_cast<uintptr_t>(d_chunk) & 7u) != 0) return SAB_ERR_INVALID_ARG;
  return write_chunk(ring, layer, 0, 0, K, V, stream, d_chunk);
}

sab_status sab_chunk_counter_add(long long* d_chunk, long long delta, void* stream) {
  if (d_chunk == nullptr || (reinterpret_cast<uintptr_t>(d_chunk) & 7u) != 0) return SAB_ERR_INVALID_ARG;
  return launch_counter_add(d_chunk, delta, static_cast<cudaStream_t>(stream)) == cudaSuccess ? SAB_OK
                                                                                            : SAB_ERR_CUDA;
}

// Allocation-free variant: the split merge goes through the library's own
// device scratch (a file-scope array of the attention kernel's translation
// unit) instead of a caller workspace.  Not a counterpart of anything in the
// method; see include/sab.h.
sab_status sab_chunk_attention_noalloc(const sab_ring* ring, int layer, long long chunk, const void* Q,
                                       const void* K_cur, const void* V_cur, int window, int use_sink,
                                       int num_splits, float softmax_scale, void* O, float* LSE, void* stream) {
  if (num_splits < 1) return SAB_ERR_INVALID_ARG;
  AttnParams p;
  const sab_status st =
      plan_chunk_attention(ring, layer, chunk, Q, K_cur, V_cur, window, use_sink, num_splits, softmax_scale, O, LSE, p);
  if (st != SAB_OK) return st;
  if (num_splits == 1) return launch_attention(p, ring->d.chunk_tokens, 1, nullptr, 0, stream);
  const WsLayout w = ws_layout(ring->d.batch * ring->d.heads, ring->d.chunk_tokens, ring->d.head_dim, num_splits);
  void* scratch = nullptr;
  size_t cap = 0;
  if (noalloc_scratch(&scratch, &cap) != cudaSuccess) return SAB_ERR_CUDA;
  if (w.total > cap) return SAB_ERR_WORKSPACE;
  // the arrival counters must start at zero; the partial rows are fully rewritten
  if (cudaMemsetAsync(scratch, 0, w.o_off, static_cast<cudaStream_t>(stream)) != cudaSuccess) return SAB_ERR_CUDA;
  return launch_attention(p, ring->d.chunk_tokens, num_splits, scratch, cap, stream);
}

size_t sab_block_causal_attention_workspace(int B, int L, int H, int D, int num_splits) {
  if (B < 1 || L < 1 || H < 1 || (D != 64 && D != 128) || num_splits < 0 || num_splits > kMaxSplits) return 0;
  if (num_splits == 0) num_splits = kMaxAutoSplits;
  return ws_layout(B * H, L, D, num_splits).total;
}

sab_status sab_block_causal_attention(const void* Q, const void* K, const void* V, int B, int L, int H, int D,
                                      int chunk_tokens, int window, int num_splits, float softmax_scale, void* O,
                                      float* LSE, void* workspace, size_t ws_bytes, void* stream) {
  if (Q == nullptr || K == nullptr || V == nullptr || O == nullptr) return SAB_ERR_INVALID_ARG;
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O)) return SAB_ERR_INVALID_ARG;
  if (LSE != nullptr && (reinterpret_cast<uintptr_t>(LSE) & 3u) != 0) return SAB_ERR_INVALID_ARG;
  if (B < 1 || L < 1 || H < 1 || (D != 64 && D != 128) || chunk_tokens < 1 || window < 0) return SAB_ERR_INVALID_ARG;
  if (num_splits < 0 || num_splits > kMaxSplits) return SAB_ERR_INVALID_ARG;
  if (!(softmax_scale > 0.f) || !isfinite(softmax_scale)) return SAB_ERR_INVALID_ARG;
  if ((long long)L > (1LL << 30)) return SAB_ERR_INVALID_ARG;
  AttnParams p;
  memset(&p, 0, sizeof(p));
  p.mode = kModeBlockCausal;
  p.B = B;
  p.H = H;
  p.D = D;
  p.scale_log2 = softmax_scale * 1.4426950408889634f;
  p.chunk_tokens = chunk_tokens;
  p.window = window;
  p.Lk = L;
  p.src_rows[0] = L;
  p.O = static_cast<uint16_t*>(O);
  p.LSE = LSE;
  if (!encode_token_major(&p.q_map, Q, B, L, H, D) || !encode_token_major(&p.k_map[0], K, B, L, H, D) ||
      !encode_token_major(&p.v_map[0], V, B, L, H, D) || !encode_token_major(&p.o_map, O, B, L, H, D))
    return SAB_ERR_CUDA;
  p.k_map[1] = p.k_map[0];
  p.v_map[1] = p.v_map[0];
  return launch_attention(p, L, num_splits, workspace, ws_bytes, stream);
}

sab_status sab_memory_prefix_attention(const void* Q, const void* K, const void* V, int B, int L, int H, int D,
                                       int mem_pad, const int* mem_len, int chunk_tokens, int window,
                                       float softmax_scale, void* O, float* LSE, void* stream) {
  if (Q == nullptr || K == nullptr || V == nullptr || O == nullptr) return SAB_ERR_INVALID_ARG;
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O)) return SAB_ERR_INVALID_ARG;
  if (LSE != nullptr && (reinterpret_cast<uintptr_t>(LSE) & 3u) != 0) return SAB_ERR_INVALID_ARG;
  if (B < 1 || L < 1 || H < 1 || (D != 64 && D != 128) || chunk_tokens < 1 || window < 0) return SAB_ERR_INVALID_ARG;
  if (mem_pad < 0 || mem_pad > L) return SAB_ERR_INVALID_ARG;
  if (mem_pad > 0 && (mem_len == nullptr || (reinterpret_cast<uintptr_t>(mem_len) & 3u) != 0))
    return SAB_ERR_INVALID_ARG;
  if (!(softmax_scale > 0.f) || !isfinite(softmax_scale)) return SAB_ERR_INVALID_ARG;
  if ((long long)L > (1LL << 30)) return SAB_ERR_INVALID_ARG;
  AttnParams p;
  memset(&p, 0, sizeof(p));
  p.mode = mem_pad > 0 ? kModeMemPrefix : kModeBlockCausal;
  p.B = B;
  p.H = H;
  p.D = D;
  p.scale_log2 = softmax_scale * 1.4426950408889634f;
  p.chunk_tokens = chunk_tokens;
  p.window = window;
  p.Lk = L;
  p.src_rows[0] = L;
  p.mem_pad = mem_pad;
  p.mem_len = mem_len;
  p.O = static_cast<uint16_t*>(O);
  p.LSE = LSE;
  if (!encode_token_major(&p.q_map, Q, B, L, H, D) || !encode_token_major(&p.k_map[0], K, B, L, H, D) ||
      !encode_token_major(&p.v_map[0], V, B, L, H, D) || !encode_token_major(&p.o_map, O, B, L, H, D))
    return SAB_ERR_CUDA;
  p.k_map[1] = p.k_map[0];
  p.v_map[1] = p.v_map[0];
  // one query tile per CTA, unsplit: the key runs are planned per CTA
  return launch_attention(p, L, 1, nullptr, 0, stream);
}

size_t sab_block_causal_attention_backward_workspace(int B, int L, int H) {
  if (B < 1 || L < 1 || H < 1) return 0;
  return align_up((size_t)B * H * L * sizeof(float), kAlign);
}

static sab_status attention_backward(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                                     const float* LSE, int B, int L, int H, int D, int mem_pad, const int* mem_len,
                                     int chunk_tokens, int window, float softmax_scale, void* dQ, void* dK, void* dV,
                                     void* workspace, size_t ws_bytes, void* stream) {
  const void* ins[] = {Q, K, V, O, dO, dQ, dK, dV};
  for (const void* x : ins)
    if (x == nullptr || !aligned16(x)) return SAB_ERR_INVALID_ARG;
  if (LSE == nullptr || (reinterpret_cast<uintptr_t>(LSE) & 3u) != 0) return SAB_ERR_INVALID_ARG;
  if (B < 1 || L < 1 || H < 1 || (D != 64 && D != 128) || chunk_tokens < 1 || window < 0) return SAB_ERR_INVALID_ARG;
  if (mem_pad < 0 || mem_pad > L) return SAB_ERR_INVALID_ARG;
  if (mem_pad > 0 && (mem_len == nullptr || (reinterpret_cast<uintptr_t>(mem_len) & 3u) != 0))
    return SAB_ERR_INVALID_ARG;
  if (!(softmax_scale > 0.f) || !isfinite(softmax_scale)) return SAB_ERR_INVALID_ARG;
  if ((long long)L > (1LL << 30) || (long long)B * H > 65535) return SAB_ERR_INVALID_ARG;
  if (workspace == nullptr || ws_bytes < sab_block_causal_attention_backward_workspace(B, L, H) ||
      (reinterpret_cast<uintptr_t>(workspace) % kAlign) != 0)
    return SAB_ERR_WORKSPACE;
  BwdParams p;
  memset(&p, 0, sizeof(p));
  p.O = static_cast<const uint16_t*>(O);
  p.dO = static_cast<const uint16_t*>(dO);
  p.LSE = LSE;
  p.delta = static_cast<float*>(workspace);
  p.dQ = static_cast<uint16_t*>(dQ);
  p.dK = static_cast<uint16_t*>(dK);
  p.dV = static_cast<uint16_t*>(dV);
  p.B = B;
  p.H = H;
  p.D = D;
  p.L = L;
  p.chunk_tokens = chunk_tokens;
  p.window = window;
  p.mem_pad = mem_pad;
  p.mem_len = mem_pad > 0 ? mem_len : nullptr;
  p.scale = softmax_scale;
  p.scale_log2 = softmax_scale * 1.4426950408889634f;
  if (!encode_token_major(&p.q_map, Q, B, L, H, D) || !encode_token_major(&p.k_map, K, B, L, H, D) ||
      !encode_token_major(&p.v_map, V, B, L, H, D) || !encode_token_major(&p.do_map, dO, B, L, H, D) ||
      !encode_token_major(&p.q_map_h, Q, B, L, H, D, 64) || !encode_token_major(&p.k_map_h, K, B, L, H, D, 64) ||
      !encode_token_major(&p.v_map_h, V, B, L, H, D, 64) || !encode_token_major(&p.do_map_h, dO, B, L, H, D, 64))
    return SAB_ERR_CUDA;
  return launch_attention_backward(p, static_cast<cudaStream_t>(stream)) == cudaSuccess ? SAB_OK : SAB_ERR_CUDA;
}

sab_status sab_block_causal_attention_backward(const void* Q, const void* K, const void* V, const void* O,
                                               const void* dO, const float* LSE, int B, int L, int H, int D,
                                               int chunk_tokens, int window, float softmax_scale, void* dQ,
                                               void* dK, void* dV, void* workspace, size_t ws_bytes,
                                               void* stream) {
  return attention_backward(Q, K, V, O, dO, LSE, B, L, H, D, 0, nullptr, chunk_tokens, window, softmax_scale, dQ, dK,
                            dV, workspace, ws_bytes, stream);
}

sab_status sab_memory_prefix_attention_backward(const void* Q, const void* K, const void* V, const void* O,
                                                const void* dO, const float* LSE, int B, int L, int H, int D,
                                                int mem_pad, const int* mem_len, int chunk_tokens, int window,
                                                float softmax_scale, void* dQ, void* dK, void* dV, void* workspace,
                                                size_t ws_bytes, void* stream) {
  return attention_backward(Q, K, V, O, dO, LSE, B, L, H, D, mem_pad, mem_len, chunk_tokens, window, softmax_scale,
                            dQ, dK, dV, workspace, ws_bytes, stream);
}

sab_status sab_selftest_split_abort(const sab_ring* ring, int layer, long long chunk, const void* Q,
                                    const void* K_cur, const void* V_cur, int window, int use_sink, int num_splits,
                                    float softmax_scale, void* O, float* LSE, void* workspace, size_t ws_bytes,
                                    int abort_split, void* stream) {
  if (num_splits < 2 || num_splits > kMaxSplits) return SAB_ERR_INVALID_ARG;
  if (abort_split < 0 || abort_split >= num_splits) return SAB_ERR_INVALID_ARG;
  AttnParams p;
  const sab_status st =
      plan_chunk_attention(ring, layer, chunk, Q, K_cur, V_cur, window, use_sink, num_splits, softmax_scale, O, LSE, p);
  if (st != SAB_OK) return st;
  p.inject_abort = abort_split + 1;
  return launch_attention(p, ring->d.chunk_tokens, num_splits, workspace, ws_bytes, stream);
}

sab_status sab_selftest_bounded_wait(unsigned long long timeout_ns, void* stream) {
  if (timeout_ns < 1000000ull || timeout_ns > 2000000000ull) return SAB_ERR_INVALID_ARG;
  return launch_wait_timeout_probe(timeout_ns, static_cast<cudaStream_t>(stream)) == cudaSuccess ? SAB_OK
                                                                                                : SAB_ERR_CUDA;
}

sab_status sab_get_last_device_error(void* stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return SAB_ERR_CUDA;
  unsigned v = 0;
  if (read_and_clear_device_error(&v) != cudaSuccess) return SAB_ERR_CUDA;
  if (v & kErrBoundsBit) return SAB_ERR_BOUNDS;
  return v ? SAB_ERR_TIMEOUT : SAB_OK;
}

int sab_debug_bounds_enabled(void) { return kDebugBounds ? 1 : 0; }

sab_status sab_debug_inject_bounds_error(int what) {
  if (!kDebugBounds) return SAB_ERR_UNSUPPORTED;
  if (what < 0 || what > SAB_DEBUG_INJECT_WS_TILE) return SAB_ERR_INVALID_ARG;
  g_inject.store(what);
  return SAB_OK;
}

const char* sab_status_string(sab_status status) {
  switch (status) {
    case SAB_OK: return "SAB_OK";
    case SAB_ERR_INVALID_ARG: return "SAB_ERR_INVALID_ARG";
    case SAB_ERR_UNSUPPORTED: return "SAB_ERR_UNSUPPORTED";
    case SAB_ERR_OUT_OF_RANGE: return "SAB_ERR_OUT_OF_RANGE";
    case SAB_ERR_WORKSPACE: return "SAB_ERR_WORKSPACE";
    case SAB_ERR_CUDA: return "SAB_ERR_CUDA";
    case SAB_ERR_TIMEOUT: return "SAB_ERR_TIMEOUT";
    case SAB_ERR_BOUNDS: return "SAB_ERR_BOUNDS";
  }
  return "SAB_ERR_UNKNOWN";
}

const char* sab_version(void) { return "sab 0.1.0 (sm_103a)"; }

}  // extern "C"
