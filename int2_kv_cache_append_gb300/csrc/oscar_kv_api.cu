// C ABI: argument validation, cache layout arithmetic and kernel dispatch.
#include <cmath>
#include <cstring>

#include "internal.h"

namespace {

using oscar::Geom;

int validate(const oscar_kv_config* c) {
  if (!c) return OSCAR_ERR_INVALID;
  if (c->num_layers <= 0 || c->batch <= 0 || c->num_q_heads <= 0 || c->num_kv_heads <= 0 ||
      c->capacity <= 0 || c->sink < 0 || c->recent < 0)
    return OSCAR_ERR_INVALID;
  if (c->num_q_heads % c->num_kv_heads != 0) return OSCAR_ERR_INVALID;
  if (!(c->k_clip > 0.f && c->k_clip <= 1.f) || !(c->v_clip > 0.f && c->v_clip <= 1.f)) return OSCAR_ERR_INVALID;
  if (c->flags & ~uint32_t(OSCAR_FLAG_ABSORB_V | OSCAR_FLAG_IN_FP32 | OSCAR_FLAG_OUT_FP32 | OSCAR_FLAG_HADAMARD |
                           OSCAR_FLAG_V_BF16 | OSCAR_FLAG_LLOYD_MAX))
    return OSCAR_ERR_INVALID;
  if (c->group_size != OSCAR_KV_GROUP) return OSCAR_ERR_UNSUPPORTED;
  if (c->head_dim != 128 && c->head_dim != 256 && c->head_dim != 512) return OSCAR_ERR_UNSUPPORTED;
  if (c->num_q_heads / c->num_kv_heads > 8) return OSCAR_ERR_UNSUPPORTED;
  return OSCAR_OK;
}

Geom make_geom(const oscar_kv_config* c) {
  Geom g;
  g.B = c->batch;
  g.Hq = c->num_q_heads;
  g.Hkv = c->num_kv_heads;
  g.D = c->head_dim;
  g.G = g.Hq / g.Hkv;
  g.Dg = g.D / OSCAR_KV_GROUP;
  g.S = c->sink;
  g.W = c->recent;
  g.cap = c->capacity;
  const int64_t n = c->capacity > c->sink ? c->capacity - c->sink : 0;
  g.ncap = (n + oscar::kNcapRound - 1) / oscar::kNcapRound * oscar::kNcapRound;
  const uint64_t bh = uint64_t(g.B) * g.Hkv;
  g.sink_bytes = oscar::align256(bh * g.S * g.D * 2);
  g.ring_bytes = oscar::align256(bh * g.W * g.D * 2);
  g.codes_bytes = oscar::align256(bh * uint64_t(g.ncap) * (g.D / 4));
  g.sz_bytes = oscar::align256(bh * uint64_t(g.ncap) * g.Dg * 4);
  g.role_bytes = g.sink_bytes + g.ring_bytes + g.codes_bytes + g.sz_bytes;
  g.vb = (c->flags & OSCAR_FLAG_V_BF16) ? 1 : 0;
  g.lm = (c->flags & OSCAR_FLAG_LLOYD_MAX) ? 1 : 0;
  g.v_role_bytes = g.vb ? oscar::align256(bh * uint64_t(g.cap) * g.D * 2) : g.role_bytes;
  g.layer_bytes = g.role_bytes + g.v_role_bytes;
  return g;
}

}  // namespace

namespace oscar {
Geom geom_of(const oscar_kv_config* c) { return make_geom(c); }
}  // namespace oscar

namespace {
bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace

namespace {

// Validates kv_append's arguments and fills *a; launches nothing.
int prep_append(const oscar_kv_config* cfg, void* cache, int32_t layer, const void* k_new, const void* v_new,
                const int32_t* start_pos, int32_t n_new, const float* R_K, const float* R_V, float* debug_rot_out,
                int32_t* dev_status, oscar::AppendArgs* a) {
  const int v = validate(cfg);
  if (v != OSCAR_OK) return v;
  // with the in-quant Hadamard the rotation matrices are not read (NULL allowed)
  const bool had = (cfg->flags & OSCAR_FLAG_HADAMARD) != 0;
  if (had) R_K = R_V = nullptr;
  if (!cache || !k_new || !v_new || !start_pos || (!had && (!R_K || !R_V))) return OSCAR_ERR_INVALID;
  if (layer < 0 || layer >= cfg->num_layers || n_new < 0) return OSCAR_ERR_INVALID;
  if (!aligned(cache, 256) || !aligned(R_K, 16) || !aligned(R_V, 16) || !aligned(k_new, 16) ||
      !aligned(v_new, 16) || (debug_rot_out && !aligned(debug_rot_out, 16)))
    return OSCAR_ERR_INVALID;
  if (n_new > cfg->capacity) return OSCAR_ERR_CAPACITY;
  a->g = make_geom(cfg);
  a->layer_base = static_cast<uint8_t*>(cache) + uint64_t(layer) * a->g.layer_bytes;
  a->k_new = k_new;
  a->v_new = v_new;
  a->start_pos = start_pos;
  a->R_K = R_K;
  a->R_V = R_V;
  a->debug_rot = debug_rot_out;
  a->status = dev_status;
  a->n_new = n_new;
  a->rows = int64_t(cfg->batch) * n_new * cfg->num_kv_heads;
  a->k_clip = cfg->k_clip;
  a->v_clip = cfg->v_clip;
  a->in_fp32 = (cfg->flags & OSCAR_FLAG_IN_FP32) ? 1 : 0;
  a->hadamard = had ? 1 : 0;
  return OSCAR_OK;
}

// Validates attn_decode's arguments and fills *a; launches nothing.
int prep_decode(const oscar_kv_config* cfg, const void* cache, int32_t layer, const void* q,
                const int32_t* seq_lens, int32_t seq_len_hint, const float* R_K, const float* R_V, float sm_scale,
                int32_t num_splits, void* out, float* lse, void* workspace, uint64_t workspace_bytes,
                int32_t* dev_status, oscar::DecodeArgs* ap) {
  oscar::DecodeArgs& a = *ap;
  const int v = validate(cfg);
  if (v != OSCAR_OK) return v;
  const bool had = (cfg->flags & OSCAR_FLAG_HADAMARD) != 0;
  if (had) R_K = R_V = nullptr;
  if (!cache || !q || !seq_lens || (!had && (!R_K || !R_V)) || !out || !workspace) return OSCAR_ERR_INVALID;
  if (layer < 0 || layer >= cfg->num_layers || num_splits < 0 || num_splits > OSCAR_KV_MAX_SPLITS ||
      seq_len_hint < 0)
    return OSCAR_ERR_INVALID;
  if (!aligned(cache, 256) || !aligned(workspace, 256) || !aligned(R_K, 16) || !aligned(R_V, 16) ||
      !aligned(q, 16) || !aligned(out, 16))
    return OSCAR_ERR_INVALID;
  if (seq_len_hint > cfg->capacity) return OSCAR_ERR_CAPACITY;
  const Geom g = make_geom(cfg);
  // the decode's TMA row coordinates are 32-bit: rows of each BF16 map must fit
  const uint64_t bhk = uint64_t(g.B) * g.Hkv;
  const uint64_t map_rows = bhk * uint64_t(g.vb ? (g.cap > g.S ? g.cap : g.S) : g.S);
  if (map_rows >= (uint64_t(1) << 31) || bhk * uint64_t(g.W) >= (uint64_t(1) << 31)) return OSCAR_ERR_UNSUPPORTED;
  const int hint = seq_len_hint > 0 ? seq_len_hint : cfg->capacity;
  // partial slots per (sequence, query head): as many as the workspace holds,
  // up to OSCAR_KV_MAX_SPLITS; an explicit split count must fit in full
  if (num_splits > 0 && oscar::decode_workspace_bytes(g, num_splits) > workspace_bytes) return OSCAR_ERR_WORKSPACE;
  int ns = OSCAR_KV_MAX_SPLITS;
  while (ns > 1 && oscar::decode_workspace_bytes(g, ns) > workspace_bytes) --ns;
  if (oscar::decode_workspace_bytes(g, ns) > workspace_bytes) return OSCAR_ERR_WORKSPACE;
  const int ctas = oscar::decode_grid(g, hint, num_splits);
  if (ctas < 1) return OSCAR_ERR_LAUNCH;

  a.g = g;
  a.layer_base = static_cast<const uint8_t*>(cache) + uint64_t(layer) * g.layer_bytes;
  a.q = q;
  a.seq_lens = seq_lens;
  a.R_K = R_K;
  a.R_V = R_V;
  a.out = out;
  a.lse = lse;
  a.status = dev_status;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const uint64_t bq = uint64_t(g.B) * g.Hq;
  const uint64_t units = uint64_t(g.B) * g.Hkv, nqt = g.G > 4 ? 2 : 1;
  a.qfrag = reinterpret_cast<uint32_t*>(ws);
  ws += oscar::align256(units * g.Dg * nqt * 2048);
  a.qbfrag = reinterpret_cast<uint32_t*>(ws);
  ws += oscar::align256(units * g.Dg * nqt * 4096);
  a.qsum = reinterpret_cast<float*>(ws);
  ws += oscar::align256(bq * g.Dg * 4);
  a.qF = reinterpret_cast<float*>(ws);
  ws += oscar::align256(bq * g.Dg * 4);
  a.ws_acc = reinterpret_cast<float*>(ws);
  ws += oscar::align256(bq * uint64_t(ns) * g.D * 4);
  a.ws_ml = reinterpret_cast<float*>(ws);
  ws += oscar::align256(bq * uint64_t(ns) * 2 * 4);
  a.ticket = reinterpret_cast<int32_t*>(ws);
  a.ns = ns;
  a.ctas = ctas;
  const float scale = sm_scale > 0.f ? sm_scale : 1.0f / std::sqrt(float(g.D));
  a.qscale = scale * 1.4426950408889634f;
  a.in_fp32 = (cfg->flags & OSCAR_FLAG_IN_FP32) ? 1 : 0;
  a.out_fp32 = (cfg->flags & OSCAR_FLAG_OUT_FP32) ? 1 : 0;
  a.absorb_v = (cfg->flags & OSCAR_FLAG_ABSORB_V) ? 1 : 0;
  a.hadamard = had ? 1 : 0;
  a.new_pos = nullptr;
  a.new_n = 0;
  a.fused = 0;
  a.wait_ns = oscar::g_test_wait_ns > 0 ? oscar::g_test_wait_ns : 2000000000ull;
  a.wait_poison = oscar::g_test_wait_poison;
  return OSCAR_OK;
}

}  // namespace

extern "C" {

int kv_layout_query(const oscar_kv_config* cfg, oscar_kv_layout* out) {
  const int v = validate(cfg);
  if (v != OSCAR_OK) return v;
  if (!out) return OSCAR_ERR_INVALID;
  const Geom g = make_geom(cfg);
  std::memset(out, 0, sizeof(*out));
  out->ncap = uint64_t(g.ncap);
  out->sink_bytes = g.sink_bytes;
  out->ring_bytes = g.ring_bytes;
  out->codes_bytes = g.codes_bytes;
  out->sz_bytes = g.sz_bytes;
  out->role_bytes = g.role_bytes;
  out->layer_bytes = g.layer_bytes;
  out->v_role_bytes = g.v_role_bytes;
  out->total_bytes = g.layer_bytes * uint64_t(cfg->num_layers);
  out->decode_workspace_bytes = oscar::decode_workspace_bytes(g, OSCAR_KV_MAX_SPLITS);
  out->max_splits = OSCAR_KV_MAX_SPLITS;
  return OSCAR_OK;
}

int kv_append(const oscar_kv_config* cfg, void* cache, int32_t layer, const void* k_new, const void* v_new,
              const int32_t* start_pos, int32_t n_new, const float* R_K, const float* R_V,
              float* debug_rot_out, int32_t* dev_status, void* stream) {
  oscar::AppendArgs a;
  const int v = prep_append(cfg, cache, layer, k_new, v_new, start_pos, n_new, R_K, R_V, debug_rot_out, dev_status, &a);
  if (v != OSCAR_OK) return v;
  return oscar::launch_append(a, static_cast<cudaStream_t>(stream));
}

int attn_decode(const oscar_kv_config* cfg, const void* cache, int32_t layer, const void* q,
                const int32_t* seq_lens, int32_t seq_len_hint, const float* R_K, const float* R_V,
                float sm_scale, int32_t num_splits, void* out, float* lse, void* workspace,
                uint64_t workspace_bytes, int32_t* dev_status, void* stream) {
  oscar::DecodeArgs a;
  const int v = prep_decode(cfg, cache, layer, q, seq_lens, seq_len_hint, R_K, R_V, sm_scale, num_splits, out, lse,
                            workspace, workspace_bytes, dev_status, &a);
  if (v != OSCAR_OK) return v;
  return oscar::launch_decode(a, static_cast<cudaStream_t>(stream));
}

int decode_step(const oscar_kv_config* cfg, void* cache, int32_t layer, const void* k_new, const void* v_new,
                const int32_t* start_pos, int32_t n_new, const void* q, const int32_t* seq_lens,
                int32_t seq_len_hint, const float* R_K, const float* R_V, float sm_scale, int32_t num_splits,
                void* out, float* lse, void* workspace, uint64_t workspace_bytes, int32_t* dev_status,
                void* stream) {
  oscar::AppendArgs aa;
  oscar::DecodeArgs ad;
  int v = prep_append(cfg, cache, layer, k_new, v_new, start_pos, n_new, R_K, R_V, nullptr, dev_status, &aa);
  if (v != OSCAR_OK) return v;
  v = prep_decode(cfg, cache, layer, q, seq_lens, seq_len_hint, R_K, R_V, sm_scale, num_splits, out, lse, workspace,
                  workspace_bytes, dev_status, &ad);
  if (v != OSCAR_OK) return v;
  // the decode kernels know what the append writes: they start streaming the
  // rest of the cache while it runs
  ad.new_pos = start_pos;
  ad.new_n = n_new;
  ad.fused = 1;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  v = oscar::launch_append(aa, st);
  if (v != OSCAR_OK) return v;
  return oscar::launch_decode(ad, st);
}

int oscar_kv_set_profile_events(void* split_start, void* split_stop) {
  oscar::g_prof_start = static_cast<cudaEvent_t>(split_start);
  oscar::g_prof_stop = static_cast<cudaEvent_t>(split_stop);
  return OSCAR_OK;
}

int oscar_kv_decode_kernels(const oscar_kv_config* cfg) {
  const int v = validate(cfg);
  if (v != OSCAR_OK) return v;
  return oscar::decode_kernel_count(make_geom(cfg), (cfg->flags & OSCAR_FLAG_ABSORB_V) != 0,
                                    (cfg->flags & OSCAR_FLAG_HADAMARD) != 0);
}

int oscar_kv_set_wait_test(uint64_t wait_ns, int32_t extra_bytes) {
  if (wait_ns > 10000000000ull || extra_bytes < 0 || extra_bytes > (1 << 20)) return OSCAR_ERR_INVALID;
  oscar::g_test_wait_ns = wait_ns;
  oscar::g_test_wait_poison = extra_bytes;
  return OSCAR_OK;
}
int oscar_calibrate_workspace_query(int32_t head_dim, uint64_t* bytes) {
  if (!bytes) return OSCAR_ERR_INVALID;
  if (head_dim != 128 && head_dim != 256 && head_dim != 512) return OSCAR_ERR_UNSUPPORTED;
  *bytes = oscar::calibrate_workspace_bytes(head_dim);
  return OSCAR_OK;
}

int oscar_calibrate_rk(const float* q, int64_t n_rows, int32_t head_dim, float* R_K_out, void* workspace,
                       uint64_t workspace_bytes, int32_t* dev_status, void* stream) {
  if (head_dim != 128 && head_dim != 256 && head_dim != 512) return OSCAR_ERR_UNSUPPORTED;
  if (!q || !R_K_out || !workspace || n_rows < 1 || n_rows > OSCAR_KV_CALIB_MAX_ROWS) return OSCAR_ERR_INVALID;
  if (!aligned(q, 16) || !aligned(R_K_out, 16) || !aligned(workspace, 256)) return OSCAR_ERR_INVALID;
  if (workspace_bytes < oscar::calibrate_workspace_bytes(head_dim)) return OSCAR_ERR_WORKSPACE;
  return oscar::launch_calibrate(q, n_rows, head_dim, R_K_out, workspace, dev_status,
                                 static_cast<cudaStream_t>(stream));
}

int oscar_calibrate_rv_workspace_query(int32_t head_dim, int64_t n_kv_rows, uint64_t* bytes) {
  if (!bytes || n_kv_rows < 1 || n_kv_rows > OSCAR_KV_CALIB_MAX_ROWS) return OSCAR_ERR_INVALID;
  if (head_dim != 128 && head_dim != 256 && head_dim != 512) return OSCAR_ERR_UNSUPPORTED;
  *bytes = oscar::calibrate_rv_workspace_bytes(head_dim, n_kv_rows);
  return OSCAR_OK;
}

int oscar_calibrate_rv(const float* q, int64_t n_q_rows, const float* k, const float* v, int64_t n_kv_rows,
                       int32_t head_dim, float* R_V_out, void* workspace, uint64_t workspace_bytes,
                       int32_t* dev_status, void* stream) {
  if (head_dim != 128 && head_dim != 256 && head_dim != 512) return OSCAR_ERR_UNSUPPORTED;
  if (!q || !k || !v || !R_V_out || !workspace) return OSCAR_ERR_INVALID;
  if (n_q_rows < 1 || n_q_rows > OSCAR_KV_CALIB_MAX_ROWS || n_kv_rows < 1 || n_kv_rows > OSCAR_KV_CALIB_MAX_ROWS)
    return OSCAR_ERR_INVALID;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(R_V_out, 16) || !aligned(workspace, 256))
    return OSCAR_ERR_INVALID;
  if (workspace_bytes < oscar::calibrate_rv_workspace_bytes(head_dim, n_kv_rows)) return OSCAR_ERR_WORKSPACE;
  return oscar::launch_calibrate_rv(q, n_q_rows, k, v, n_kv_rows, head_dim, R_V_out, workspace, dev_status,
                                    static_cast<cudaStream_t>(stream));
}

}  // extern "C"
