// Internal interface between the host API (sab_api.cu) and the kernels.
// Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace sab {

constexpr int kTileM = 128;    // query rows per tile (one TMEM lane per row)
constexpr int kTileN = 128;    // keys per KV tile
constexpr int kMaxSegments = 4;

// One contiguous run of key rows inside one K/V source.
//   src 0: the layer's ring (rows along the [B,H,rows,D] row axis),
//   src 1: the current chunk passed in (token axis of [B,L,H,D]).
struct KvSegment {
  int src;
  int row0;    // first row of the run in the source's row axis
  int nrows;   // rows in the run
  int tile0;   // global index of the run's first 128-key tile
};

enum AttnMode : int { kModeStreaming = 0, kModeBlockCausal = 1 };

struct AttnParams {
  CUtensorMap q_map;      // dims (D, Lq, H, B), box (64, 128, 1, 1), SW128
  CUtensorMap k_map[2];   // per source, dims (D, rows, H, B)
  CUtensorMap v_map[2];
  CUtensorMap o_map;      // output, dims (D, Lq, H, B), box (64, 128, 1, 1), SW128
  int mode;
  int fp8;                // 1: the ring holds 8-bit codes (k_map[0]/v_map[0] are uint8 maps)
  int k_int8;             // with fp8: keys are INT8 codes (values stay E4M3)
  const float* k_scale;   // FP8: [B*H][scale_stride] fp32 scales, index = ring row / chunk_tokens
  const float* v_scale;
  int scale_stride;
  int B, H, D;
  int Lq;                 // query rows per (b, h)
  int n_qtiles;           // ceil(Lq / 128)
  int n_qgroups;          // CTAs along the query axis (q tiles per CTA: 1 or 2)
  int lq_pad;             // n_qgroups * tiles per CTA * 128 (workspace row pitch)
  int splits;
  int cluster_merge;      // 0: splits merge through the workspace; 1: the splits
                          // of a query group form a thread-block cluster and
                          // merge through distributed shared memory; 2: two
                          // splits of a two-tile group merge as a CTA pair
                          // (one bulk copy each way)
  float scale_log2;       // softmax_scale * log2(e)
  // streaming
  int nseg;
  int total_tiles;
  KvSegment seg[kMaxSegments];
  // block-causal
  int chunk_tokens;
  int window;
  int Lk;
  // outputs
  uint16_t* O;            // bf16 [B, Lq, H, D]
  float* LSE;             // [B, H, Lq] or null
  // split workspace
  float* ws_o;            // [splits][B*H][lq_pad][D]
  float* ws_lse;          // [splits][B*H][lq_pad]
  unsigned int* ws_count; // [B*H][n_qgroups]
};

// FP8 append: per (b, h) block of one chunk.
struct AppendParams {
  const uint16_t* src[2];   // K, V token-major [B, Lc, H, D] bf16
  void* dst[2];             // ring K, V region base of the layer
  float* scale[2];          // FP8 only: ring K, V scale base of the layer
  int B, H, D, Lc;
  int rows;                 // rows per (b, h) in the ring
  int slot_row0;            // first row of the destination slot
  int scale_idx;            // (has_sink + slot) or 0 for the sink
  int scale_stride;         // has_sink + R
  int k_int8;               // 8-bit ring: K as INT8 (amax / 127) instead of E4M3
};

// Launchers (return cudaError_t of the launch).
cudaError_t launch_append_bf16(const AppendParams& p, cudaStream_t s);
cudaError_t launch_append_fp8(const AppendParams& p, cudaStream_t s);
cudaError_t launch_chunk_attention(const AttnParams& p, int q_tiles_per_cta, cudaStream_t s);
// One query tile per CTA, key-half softmax warpgroups; unsplit KV only.
cudaError_t launch_chunk_attention_kh(const AttnParams& p, cudaStream_t s);
cudaError_t read_and_clear_device_error(unsigned int* value);
// Device address and size of the library's own split-merge scratch.
cudaError_t noalloc_scratch(void** ptr, size_t* bytes);
int attention_q_tiles_per_cta(int D);

}  // namespace sab
