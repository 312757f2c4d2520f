// Host-side launch interface shared by the C-ABI translation unit and the
// kernel translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace oscar {

struct AppendArgs {
  Geom g;
  uint8_t* layer_base;   // cache + layer * layer_bytes
  const void* k_new;
  const void* v_new;
  const int32_t* start_pos;
  const float* R_K;
  const float* R_V;
  float* debug_rot;
  int32_t* status;
  int n_new;
  int64_t rows;          // B * n_new * Hkv
  float k_clip, v_clip;
  int in_fp32;
  int hadamard;          // rotate by the in-quant Hadamard (R_K, R_V unused)
  FastDiv div_hkv, div_n_new;  // set by the tensor-core launcher (rows < 2^31)
};

struct DecodeArgs {
  Geom g;
  const uint8_t* layer_base;
  const void* q;
  const int32_t* seq_lens;
  const float* R_K;
  const float* R_V;
  void* out;
  float* lse;
  int32_t* status;
  uint32_t* qfrag;  // [B*Hkv][Dg][NQT*512]  mma B fragments of q' (fp16 hi/lo, scaled per head)
  uint32_t* qbfrag; // [B*Hkv][Dg][NQT*1024] bf16 three-way B fragments of q', shared-memory image
  float* qsum;      // [B][Hq][Dg]  per-group sums of q' (log2 units)
  float* qF;        // [B][Hq][Dg]  score factor 2^(24 - X) of the scaled fragments
  float* ws_acc;   // [B][Hq][NS][D]
  float* ws_ml;    // [B][Hq][NS][2]
  int32_t* ticket; // [B][Hkv] split-completion counters (zeroed by qrot)
  const int32_t* new_pos;  // with fused = 1: positions [new_pos[b], new_pos[b] + new_n) are being
  int new_n;               // written by the preceding append kernel of the same call
  int fused;
  int ns;          // partial slots per (b, query head) in the workspace
  int ctas;        // CTAs of the split kernel
  float qscale;    // sm_scale * log2(e)
  int in_fp32, out_fp32, absorb_v;
  int hadamard;    // q and the output use the in-quant Hadamard (R_K, R_V unused)
  uint64_t wait_ns;  // limit of every barrier wait in the split kernel (test hook; ~2 s by default)
  int wait_poison;   // test hook: extra bytes CTA 0 expects on its first copy (0 normally)
};

uint64_t decode_workspace_bytes(const Geom& g, int ns);
// kernels one attn_decode launches
int decode_kernel_count(const Geom& g, bool absorb_v, bool hadamard);
// cache geometry of a validated configuration
Geom geom_of(const oscar_kv_config* c);
// optional events recorded around the split kernel (per host thread)
extern thread_local cudaEvent_t g_prof_start, g_prof_stop;
// timeout-path test hook (per host thread): wait limit and extra expected bytes
extern thread_local uint64_t g_test_wait_ns;
extern thread_local int g_test_wait_poison;
int launch_append(const AppendArgs& a, cudaStream_t stream);
int launch_append_tc(const AppendArgs& a, cudaStream_t stream);  // D = 128, bf16 inputs
// 2-D tiled TMA map of a row-major bf16 matrix [rows][cols], 128-byte swizzle
bool encode_rows_bf16(CUtensorMap* m, const void* ptr, uint64_t rows, uint32_t cols, uint32_t box_cols,
                      uint32_t box_rows);
// 2-D tiled TMA map of a row-major float32 matrix [rows][cols], no swizzle
bool encode_f32_tiles(CUtensorMap* m, const float* ptr, uint64_t rows, uint64_t cols, uint32_t box_cols,
                      uint32_t box_rows);
// 2-D tiled TMA map of INT2 code rows [rows][rowb] (uint8; rowb = 32, 64 or
// 128), box [box_rows][rowb], swizzled by the row size: 16-byte chunk c of
// row t lands at chunk c ^ ((t * rowb / 128) mod (rowb / 16))
bool encode_code_rows(CUtensorMap* m, const void* ptr, uint64_t rows, uint32_t rowb, uint32_t box_rows);
int launch_decode(const DecodeArgs& a, cudaStream_t stream);
// CTAs of the split kernel: num_splits * B * Hkv, or (num_splits = 0) as many
// as are resident at once, fewer when a context of seq_len_hint is short.
int decode_grid(const Geom& g, int seq_len_hint, int num_splits);
// R_K calibration (calibrate.cu)
uint64_t calibrate_workspace_bytes(int D);
int launch_calibrate(const float* q, int64_t n, int D, float* R, void* ws, int32_t* status, cudaStream_t stream);
// R_V calibration from the score-weighted V covariance (calibrate.cu)
uint64_t calibrate_rv_workspace_bytes(int D, int64_t n_kv);
int launch_calibrate_rv(const float* q, int64_t nq, const float* k, const float* v, int64_t nkv, int D, float* R,
                        void* ws, int32_t* status, cudaStream_t stream);

}  // namespace oscar
