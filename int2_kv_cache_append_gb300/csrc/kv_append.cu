// kv_append: rotate new K/V rows by the layer's orthogonal matrix, clip each
// row, quantise groups of 128 channels to 2-bit codes with fp16 scale/zero and
// write the BF16 sink / recent-window copies.
//
// Source: "OSCAR-LLAMACPP-Qwen3-4B-Thinking-2507-INT2-KV" model card (Files
// note: K and V are rotated orthogonally after RoPE; Run: per-row clip ratio,
// high-precision sink/recent tokens) and "OSCAR-RotationZoo" (Available
// rotations: group 128 along head_dim; How to use: K/V clip 0.96/0.92).
//
// Three CUDA-core kernels (the tensor-core kernel for large head_dim-128 bf16
// appends is in kv_append_tc.cu):
//
// kv_append_kernel, tiled: one CTA of 128 threads handles RPC = 64*128/D rows
// of one role (K or V):
//   1. stage the input rows in shared memory as float32;
//   2. rotate: each row's D outputs are split over 128/RPC threads, each
//      accumulating 32 columns at a time with fp32 FMAs (R is read through the
//      L1 as warp-wide broadcasts);
//   3. quantise: one thread per row, the row held in padded shared memory.
//
// kv_append_rows_kernel, row-parallel, for appends of a few rows (a decode
// step appends one token per sequence): 4 or 8 rows per CTA, described below.
// It also takes every append of the in-quant Hadamard mode (rows transformed
// in registers, no matrix), of the K-only INT2 mode (V rows stored as BF16
// at their positions) and of the Lloyd-Max levels (span 2 rho + 1, codes by
// comparison with the level midpoints, lm_code).
//
// kv_append_slices_kernel, the row-parallel append at head_dim 256 / 512 for
// up to 1024 rows per role: a thread-block cluster of one CTA per quant group
// shares a few rows, each CTA streaming only its column slice of R (below).
//
// All three accumulate each rotated value with fp32 FMAs in increasing
// input-channel order and run the same codec operations, so they write
// identical bytes.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"

namespace oscar {
namespace {

constexpr int kAppendThreads = 128;
// appends of at most this many rows per role take the row-parallel kernel
constexpr int64_t kSmallAppendRows = 1024;

template <int D>
struct AppendCfg {
  // rows per CTA: 64 KB of shared memory for inputs and rotated rows, so that
  // three CTAs share an SM (the rotation is fp32 FMA work that needs the warps)
  static constexpr int RPC = kAppendThreads * 64 / D;
  static constexpr int TPR = kAppendThreads / RPC;      // threads per row while rotating
  static constexpr int LD = D + 1;                      // padded smem row (conflict-free)
  static constexpr int SMEM = 2 * RPC * LD * 4;
};

// Channel held by 2-bit slot s (0..15) of word w (0..7) of a 128-channel group.
__device__ __forceinline__ int slot_channel(int role, int w, int s) {
  if (role == 0) {
    const int c = w >> 1, i = w & 1, p = s & 7, odd = s >> 3;
    const int kk = 4 * i + (p >> 1), h = p & 1;
    return 16 * kk + 2 * c + 8 * h + odd;
  }
  return 8 * s + w;
}

template <int D>
__global__ void __launch_bounds__(kAppendThreads) kv_append_kernel(const AppendArgs a) {
  using C = AppendCfg<D>;
  extern __shared__ float smem[];
  float* xs = smem;                 // [RPC][LD] inputs
  float* rs = smem + C::RPC * C::LD;  // [RPC][LD] rotated rows

  pdl_trigger();  // a dependent kernel may be scheduled now; it waits for our completion itself
  const int role = blockIdx.y;
  const float* __restrict__ R = role ? a.R_V : a.R_K;
  const float ratio = role ? a.v_clip : a.k_clip;
  const int64_t row0 = int64_t(blockIdx.x) * C::RPC;

  // 1. stage inputs (coalesced: consecutive rows are contiguous)
  if (a.in_fp32) {
    const float* src = static_cast<const float*>(role ? a.v_new : a.k_new);
    for (int idx = threadIdx.x; idx < C::RPC * D; idx += kAppendThreads) {
      const int r = idx / D, d = idx % D;
      const int64_t row = row0 + r;
      xs[r * C::LD + d] = row < a.rows ? src[row * D + d] : 0.f;
    }
  } else {
    const __nv_bfloat16* src = static_cast<const __nv_bfloat16*>(role ? a.v_new : a.k_new);
    for (int idx = threadIdx.x; idx < C::RPC * D; idx += kAppendThreads) {
      const int r = idx / D, d = idx % D;
      const int64_t row = row0 + r;
      xs[r * C::LD + d] = row < a.rows ? __bfloat162float(src[row * D + d]) : 0.f;
    }
  }
  __syncthreads();

  // 2. rotate: r_j = sum_i x_i R[i][j]
  {
    const int r = threadIdx.x % C::RPC, part = threadIdx.x / C::RPC;
    constexpr int COLS = D / C::TPR;
    const float* xrow = xs + r * C::LD;
    for (int c0 = part * COLS; c0 < (part + 1) * COLS; c0 += 32) {
      float acc[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) acc[j] = 0.f;
      const float4* Rcol = reinterpret_cast<const float4*>(R + c0);
#pragma unroll 2
      for (int i = 0; i < D; ++i) {
        const float xv = xrow[i];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const float4 rv = __ldg(Rcol + (size_t)i * (D / 4) + q);
          acc[4 * q + 0] = fmaf(xv, rv.x, acc[4 * q + 0]);
          acc[4 * q + 1] = fmaf(xv, rv.y, acc[4 * q + 1]);
          acc[4 * q + 2] = fmaf(xv, rv.z, acc[4 * q + 2]);
          acc[4 * q + 3] = fmaf(xv, rv.w, acc[4 * q + 3]);
        }
      }
#pragma unroll
      for (int j = 0; j < 32; ++j) rs[r * C::LD + c0 + j] = acc[j];
    }
  }
  __syncthreads();

  // 3. quantise one row per thread
  if (threadIdx.x >= C::RPC) return;
  const int64_t row = row0 + threadIdx.x;
  if (row >= a.rows) return;
  const Geom& g = a.g;
  const int h = int(row % g.Hkv);
  const int64_t bt = row / g.Hkv;
  const int t = int(bt % a.n_new);
  const int b = int(bt / a.n_new);
  const int p = a.start_pos[b] + t;
  const int newlen = a.start_pos[b] + a.n_new;
  const float* rr = rs + threadIdx.x * C::LD;

  if (a.debug_rot) {
    float4* dst = reinterpret_cast<float4*>(a.debug_rot + (row * 2 + role) * D);
#pragma unroll 4
    for (int d = 0; d < D; d += 4) dst[d / 4] = make_float4(rr[d], rr[d + 1], rr[d + 2], rr[d + 3]);
  }
  if (p < 0 || p >= g.cap) {
    status_or(a.status, OSCAR_DEV_OVER_CAPACITY);
    return;
  }

  uint8_t* role_base = a.layer_base + role * g.role_bytes;
  const int64_t bh = int64_t(b) * g.Hkv + h;

  // row max |r| and finiteness
  float amax = 0.f;
  bool finite = true;
  for (int d = 0; d < D; ++d) {
    const float v = rr[d];
    finite &= isfinite(v);
    amax = fmaxf(amax, fabsf(v));
  }
  if (!finite) status_or(a.status, OSCAR_DEV_NONFINITE);
  const float tclip = __fmul_rn(ratio, amax);

  // BF16 window copies of the rotated row
  const bool to_sink = p < g.S;
  const bool to_ring = g.W > 0 && p >= newlen - g.W;
  if (to_sink || to_ring) {
    uint8_t* dst = to_sink ? role_base + (bh * g.S + p) * (2 * D)
                           : role_base + g.sink_bytes + (bh * g.W + (p % g.W)) * (2 * D);
    uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll 2
    for (int d = 0; d < D; d += 8) {
      uint4 v;
      v.x = pack_bf162(__float2bfloat16_rn(rr[d + 0]), __float2bfloat16_rn(rr[d + 1]));
      v.y = pack_bf162(__float2bfloat16_rn(rr[d + 2]), __float2bfloat16_rn(rr[d + 3]));
      v.z = pack_bf162(__float2bfloat16_rn(rr[d + 4]), __float2bfloat16_rn(rr[d + 5]));
      v.w = pack_bf162(__float2bfloat16_rn(rr[d + 6]), __float2bfloat16_rn(rr[d + 7]));
      d4[d / 8] = v;
    }
    if (to_sink && to_ring) {  // p < S and inside the recent window: both copies
      uint4* r4 = reinterpret_cast<uint4*>(role_base + g.sink_bytes + (bh * g.W + (p % g.W)) * (2 * D));
      for (int d = 0; d < D; d += 8) r4[d / 8] = d4[d / 8];
    }
  }
  if (to_sink) return;  // positions < S have no INT2 row

  const int64_t irow = bh * g.ncap + (p - g.S);
  uint32_t* codes = reinterpret_cast<uint32_t*>(role_base + g.sink_bytes + g.ring_bytes + irow * (D / 4));
  uint32_t* sz = reinterpret_cast<uint32_t*>(role_base + g.sink_bytes + g.ring_bytes + g.codes_bytes) +
                 irow * (D / kGroup);

  for (int j = 0; j < D / kGroup; ++j) {
    const float* xg = rr + j * kGroup;
    float mn = INFINITY, mx = -INFINITY;
    for (int d = 0; d < kGroup; ++d) {
      const float x = fminf(fmaxf(xg[d], -tclip), tclip);
      mn = fminf(mn, x);
      mx = fmaxf(mx, x);
    }
    const float s32 = __fdiv_rn(__fsub_rn(mx, mn), 3.0f);
    const __half sh = __float2half_rn(s32);
    const __half zh = __float2half_rn(mn);
    const float sf = __half2float(sh), zf = __half2float(zh);
    const bool rng_ok = isfinite(sf) && isfinite(zf);
    if (!rng_ok) status_or(a.status, OSCAR_DEV_FP16_RANGE);
    const bool ok = rng_ok && sf != 0.f;
    const float inv = ok ? __frcp_rn(sf) : 0.f;
    uint32_t words[8];
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      uint32_t word = 0;
#pragma unroll
      for (int s = 0; s < 16; ++s) {
        const float x = fminf(fmaxf(xg[slot_channel(role, w, s)], -tclip), tclip);
        int c = __float2int_rn(__fmul_rn(__fsub_rn(x, zf), inv));
        c = ok ? min(max(c, 0), 3) : 0;
        word |= uint32_t(c) << (2 * s);
      }
      words[w] = word;
    }
    uint4* c4 = reinterpret_cast<uint4*>(codes + 8 * j);
    c4[0] = make_uint4(words[0], words[1], words[2], words[3]);
    c4[1] = make_uint4(words[4], words[5], words[6], words[7]);
    sz[j] = pack_half2(sh, zh);
  }
}

// ---------------------------------------------------------------------------
// Row-parallel variant for small appends (decode: one or a few new tokens per
// sequence).  The tiled kernels above amortise loading R over many rows and pay
// a long serial prologue; with a few dozen rows that prologue is the whole cost.
// Here each CTA takes only RPC rows of one role, so many CTAs share the work:
//   1. thread 0 streams R into shared memory in 64 KB chunks (cp.async.bulk,
//      two stages when R is larger than one chunk) while all threads stage the
//      RPC input rows transposed ([D][RPC], so one channel of all rows is one
//      broadcast load);
//   2. thread t accumulates output columns t, t + 128, ... of all RPC rows with
//      fp32 FMAs in increasing input-channel order (the same sums, in the same
//      order, as the tiled CUDA-core kernel, so results are bit-identical);
//   3. each warp quantises whole rows: lanes hold channels lane + 32e, row and
//      group extrema come from warp reductions (max/min are exact in any
//      order), and every 2-bit word is built by 32 / (8 * D/128) lanes that
//      OR their slots together.
// Waits on the copies are bounded; on a timeout the CTA flags
// OSCAR_DEV_TIMEOUT, waits (bounded) for its copies in flight and returns.
// With V kept BF16 (K-only INT2) the V rows are stored as BF16 at their
// positions instead of quantised.
// With HAD (the in-quant Hadamard) steps 1 and 2 are replaced: each warp loads
// its rows and transforms every 128-channel group in registers
// (hadamard128_warp); no rotation matrix is read.
// ---------------------------------------------------------------------------
template <int D, int RPC>
struct RowsCfg {
  static constexpr int CH_ROWS = (65536 / (D * 4)) < D ? 65536 / (D * 4) : D;  // rows of R per chunk
  static constexpr int NCH = D / CH_ROWS;
  // two stages: deeper staging (six 32 KB chunks, one CTA per SM) made the
  // head_dim-512 decode step slower, its CTAs keeping the attention kernel,
  // launched early, off their SMs
  static constexpr int NSTG = NCH > 1 ? 2 : 1;
  static constexpr uint32_t CH_BYTES = uint32_t(CH_ROWS) * D * 4;
  static constexpr int CPT = D / 128;  // output columns per thread
  static constexpr uint32_t OFF_X = NSTG * CH_BYTES;
  static constexpr uint32_t OFF_Y = OFF_X + uint32_t(D) * RPC * 4;
  static constexpr uint32_t OFF_BAR = OFF_Y + uint32_t(RPC) * D * 4;
  static constexpr uint32_t SMEM = OFF_BAR + 8 * NSTG;
  static constexpr uint32_t SMEM_HAD = uint32_t(RPC) * D * 4;  // rotated rows only
  static constexpr int NW = 8 * (D / kGroup);  // 32-bit code words per row
  static constexpr int LPW = 32 / NW;          // lanes per word
  static constexpr int SPL = 16 / LPW;         // 2-bit slots per lane
  static_assert(RPC % 4 == 0, "rows per CTA must be a multiple of the warp count");
  static_assert(SMEM <= 227 * 1024, "dynamic shared memory of one CTA");
};

// Steps 1 and 2 with a rotation matrix R: stream R into shared memory, stage
// the inputs transposed and accumulate ys = x R.  Returns false after a
// timed-out copy (OSCAR_DEV_TIMEOUT flagged, copies in flight drained).
template <int D, int RPC>
__device__ __forceinline__ bool rotate_by_matrix(const AppendArgs& a, unsigned char* sm, float* ys, int role,
                                                 int64_t row0, int tid) {
  using C = RowsCfg<D, RPC>;
  float* Rs = reinterpret_cast<float*>(sm);
  float* xs = reinterpret_cast<float*>(sm + C::OFF_X);  // [D][RPC]
  const uint32_t bar0 = smem_u32(sm + C::OFF_BAR);
  const float* __restrict__ R = role ? a.R_V : a.R_K;

  if (tid == 0) {
    for (int s = 0; s < C::NSTG; ++s) mbar_init(bar0 + 8 * s, 1);
    mbar_fence_init();
    for (int s = 0; s < C::NSTG; ++s) {
      mbar_arrive_expect_tx(bar0 + 8 * s, C::CH_BYTES);
      bulk_g2s(smem_u32(Rs) + s * C::CH_BYTES, R + size_t(s) * C::CH_ROWS * D, C::CH_BYTES, bar0 + 8 * s);
    }
  }
  // stage inputs transposed; rows past the end are zero
  for (int idx = tid; idx < RPC * D; idx += kAppendThreads) {
    const int r = idx / D, i = idx % D;
    const int64_t row = row0 + r;
    float v = 0.f;
    if (row < a.rows)
      v = a.in_fp32 ? static_cast<const float*>(role ? a.v_new : a.k_new)[row * D + i]
                    : __bfloat162float(static_cast<const __nv_bfloat16*>(role ? a.v_new : a.k_new)[row * D + i]);
    xs[i * RPC + r] = v;
  }
  __syncthreads();

  float acc[RPC][C::CPT];
#pragma unroll
  for (int r = 0; r < RPC; ++r)
#pragma unroll
    for (int m = 0; m < C::CPT; ++m) acc[r][m] = 0.f;

  bool abort = false;
  int ch = 0;
  for (; ch < C::NCH; ++ch) {
    const int s = ch % C::NSTG;
    const bool ok = mbar_wait(bar0 + 8 * s, (ch / C::NSTG) & 1);
    if (__syncthreads_or(!ok)) {
      abort = true;
      break;
    }
    const float* Rc = Rs + size_t(s) * C::CH_ROWS * D;
#pragma unroll 4
    for (int kk = 0; kk < C::CH_ROWS; ++kk) {
      const int k = ch * C::CH_ROWS + kk;
      float xv[RPC];
#pragma unroll
      for (int r4 = 0; r4 < RPC / 4; ++r4) {
        const float4 x4 = *reinterpret_cast<const float4*>(xs + k * RPC + 4 * r4);
        xv[4 * r4 + 0] = x4.x;
        xv[4 * r4 + 1] = x4.y;
        xv[4 * r4 + 2] = x4.z;
        xv[4 * r4 + 3] = x4.w;
      }
#pragma unroll
      for (int m = 0; m < C::CPT; ++m) {
        const float rv = Rc[kk * D + tid + 128 * m];
#pragma unroll
        for (int r = 0; r < RPC; ++r) acc[r][m] = fmaf(xv[r], rv, acc[r][m]);
      }
    }
    __syncthreads();  // every thread is done with stage s
    if (tid == 0 && ch + C::NSTG < C::NCH) {
      mbar_arrive_expect_tx(bar0 + 8 * s, C::CH_BYTES);
      bulk_g2s(smem_u32(Rs) + s * C::CH_BYTES, R + size_t(ch + C::NSTG) * C::CH_ROWS * D, C::CH_BYTES,
               bar0 + 8 * s);
    }
  }
  if (abort) {
    if (tid == 0) {
      status_or(a.status, OSCAR_DEV_TIMEOUT);
      // chunks issued but not consumed: ch .. min(ch + NSTG, NCH) - 1
      for (int c2 = ch; c2 < C::NCH && c2 < ch + C::NSTG; ++c2)
        (void)mbar_wait(bar0 + 8 * (c2 % C::NSTG), (c2 / C::NSTG) & 1);
    }
    return false;
  }
#pragma unroll
  for (int r = 0; r < RPC; ++r)
#pragma unroll
    for (int m = 0; m < C::CPT; ++m) ys[r * D + tid + 128 * m] = acc[r][m];
  __syncthreads();
  return true;
}

template <int D, int RPC, bool HAD>
__global__ void __launch_bounds__(kAppendThreads) kv_append_rows_kernel(const AppendArgs a) {
  using C = RowsCfg<D, RPC>;
  extern __shared__ __align__(128) unsigned char sm[];
  float* ys = reinterpret_cast<float*>(sm + (HAD ? 0 : C::OFF_Y));  // [RPC][D] rotated rows

  // Launched with programmatic dependent launch, so the CTAs can be resident
  // before the preceding kernel ends (a decode step's append follows the
  // previous layer's attention); nothing is read before the wait, and the
  // dependents (qrot) are released only after it, so they never run ahead of
  // the kernel that produced this call's inputs.
  pdl_wait();
  pdl_trigger();
  const int role = blockIdx.y;
  const int64_t row0 = int64_t(blockIdx.x) * RPC;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;

  if constexpr (HAD) {
    for (int r = warp; r < RPC; r += kAppendThreads / 32) {
      const int64_t row = row0 + r;
      if (row >= a.rows) break;
#pragma unroll
      for (int j = 0; j < D / kGroup; ++j) {
        float x[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int64_t i = row * D + j * kGroup + lane + 32 * e;
          x[e] = a.in_fp32 ? static_cast<const float*>(role ? a.v_new : a.k_new)[i]
                           : __bfloat162float(static_cast<const __nv_bfloat16*>(role ? a.v_new : a.k_new)[i]);
        }
        hadamard128_warp(x, lane);
#pragma unroll
        for (int e = 0; e < 4; ++e) ys[r * D + j * kGroup + lane + 32 * e] = x[e];
      }
    }
    __syncthreads();
  } else {
    if (!rotate_by_matrix<D, RPC>(a, sm, ys, role, row0, tid)) return;
  }

  const float ratio = role ? a.v_clip : a.k_clip;
  const Geom& g = a.g;
  uint8_t* role_base = a.layer_base + role * g.role_bytes;
  for (int r = warp; r < RPC; r += kAppendThreads / 32) {
    const int64_t row = row0 + r;
    if (row >= a.rows) break;
    const float* y = ys + r * D;
    if (a.debug_rot) {
      float* dst = a.debug_rot + (row * 2 + role) * D;
      for (int d = lane; d < D; d += 32) dst[d] = y[d];
    }
    const int h = int(row % g.Hkv);
    const int64_t bt = row / g.Hkv;
    const int t = int(bt % a.n_new);
    const int b = int(bt / a.n_new);
    const int p = a.start_pos[b] + t;
    const int newlen = a.start_pos[b] + a.n_new;
    if (p < 0 || p >= g.cap) {
      if (lane == 0) status_or(a.status, OSCAR_DEV_OVER_CAPACITY);
      continue;
    }
    const int64_t bh = int64_t(b) * g.Hkv + h;

    float v[D / 32];
    float amax = 0.f;
    bool finite = true;
#pragma unroll
    for (int e = 0; e < D / 32; ++e) {
      v[e] = y[lane + 32 * e];
      finite &= isfinite(v[e]);
      amax = fmaxf(amax, fabsf(v[e]));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    finite = __all_sync(0xffffffffu, finite);
    if (!finite && lane == 0) status_or(a.status, OSCAR_DEV_NONFINITE);
    const float tclip = __fmul_rn(ratio, amax);

    if (role == 1 && g.vb) {  // K-only INT2: the V row is kept BF16 at its position
      __nv_bfloat16* dv = reinterpret_cast<__nv_bfloat16*>(role_base + (bh * g.cap + p) * (2 * D));
#pragma unroll
      for (int e = 0; e < D / 32; ++e) dv[lane + 32 * e] = __float2bfloat16_rn(v[e]);
      continue;
    }
    const bool to_sink = p < g.S;
    const bool to_ring = g.W > 0 && p >= newlen - g.W;
    if (to_sink || to_ring) {
      __nv_bfloat16* d0 = reinterpret_cast<__nv_bfloat16*>(
          to_sink ? role_base + (bh * g.S + p) * (2 * D) : role_base + g.sink_bytes + (bh * g.W + (p % g.W)) * (2 * D));
      __nv_bfloat16* d1 = (to_sink && to_ring)
                              ? reinterpret_cast<__nv_bfloat16*>(role_base + g.sink_bytes + (bh * g.W + (p % g.W)) * (2 * D))
                              : nullptr;
#pragma unroll
      for (int e = 0; e < D / 32; ++e) {
        const __nv_bfloat16 bv = __float2bfloat16_rn(v[e]);
        d0[lane + 32 * e] = bv;
        if (d1) d1[lane + 32 * e] = bv;
      }
    }
    if (to_sink) continue;

    // group statistics; each lane keeps those of the group its code word lies in
    const int wi = lane / C::LPW, part = lane % C::LPW;
    const int my_j = wi / 8, my_w = wi % 8;
    float my_zf = 0.f, my_inv = 0.f;
    bool my_ok = false;
    uint32_t my_sz = 0;
#pragma unroll
    for (int j = 0; j < D / kGroup; ++j) {
      float mn = INFINITY, mx = -INFINITY;
#pragma unroll
      for (int e = 4 * j; e < 4 * j + 4; ++e) {
        const float x = fminf(fmaxf(v[e], -tclip), tclip);
        mn = fminf(mn, x);
        mx = fmaxf(mx, x);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      }
      const float s32 = __fdiv_rn(__fsub_rn(mx, mn), g.lm ? kLmSpan : 3.0f);
      const __half sh = __float2half_rn(s32);
      const __half zh = __float2half_rn(mn);
      const float sf = __half2float(sh), zf = __half2float(zh);
      const bool rng_ok = isfinite(sf) && isfinite(zf);
      if (!rng_ok && lane == 0) status_or(a.status, OSCAR_DEV_FP16_RANGE);
      const bool ok = rng_ok && sf != 0.f;
      if (j == my_j) {
        my_zf = zf;
        my_inv = ok ? __frcp_rn(sf) : 0.f;
        my_ok = ok;
      }
      if (lane == j) my_sz = pack_half2(sh, zh);
    }
    const int64_t irow = bh * g.ncap + (p - g.S);
    uint32_t* codes = reinterpret_cast<uint32_t*>(role_base + g.sink_bytes + g.ring_bytes + irow * (D / 4));
    uint32_t* sz = reinterpret_cast<uint32_t*>(role_base + g.sink_bytes + g.ring_bytes + g.codes_bytes) +
                   irow * (D / kGroup);
    uint32_t word = 0;
#pragma unroll
    for (int k = 0; k < C::SPL; ++k) {
      const int s = part * C::SPL + k;
      const float x = fminf(fmaxf(y[my_j * kGroup + slot_channel(role, my_w, s)], -tclip), tclip);
      const float yq = __fmul_rn(__fsub_rn(x, my_zf), my_inv);
      int c = g.lm ? lm_code(yq) : min(max(__float2int_rn(yq), 0), 3);
      c = my_ok ? c : 0;
      word |= uint32_t(c) << (2 * s);
    }
#pragma unroll
    for (int o = 1; o < C::LPW; o <<= 1) word |= __shfl_xor_sync(0xffffffffu, word, o);
    if (part == 0) codes[wi] = word;
    if (lane < D / kGroup) sz[lane] = my_sz;
  }
}

// ---------------------------------------------------------------------------
// Row-parallel append at head_dim 256 / 512, sliced by quant group.  A CTA of
// the row-parallel kernel above streams all of R through shared memory (1 MB
// at head_dim 512) for a handful of rows, so a decode step's append waits on
// that stream.  Here a thread-block cluster of D/128 CTAs shares RPC rows:
// CTA q computes output channels [128 q, 128 q + 128) — one quant group — and
// streams only that column slice of R (TMA tensor loads of 64 x 128 fp32
// boxes, 32 KB each).  The row's max |y| (the clip threshold) is the one value
// the group needs from the others: each CTA posts its slice's maximum in
// shared memory and reads the others' through distributed shared memory
// between two cluster barriers.  The rotated values are the same fp32 sums
// in the same order as in the kernels above and the codec takes the same
// operations, so the bytes written are identical.  Every CTA reaches both
// cluster barriers, also after a timed-out copy.
// ---------------------------------------------------------------------------
template <int D, int RPC>
struct SliceCfg {
  static constexpr int SL = D / kGroup;        // CTAs per cluster
  static constexpr int CH_ROWS = 64;           // rows of R's slice per chunk
  static constexpr int NCH = D / CH_ROWS;
  static constexpr int NSTG = 2;
  static constexpr uint32_t CH_BYTES = uint32_t(CH_ROWS) * kGroup * 4;
  static constexpr uint32_t OFF_X = NSTG * CH_BYTES;                  // [D][RPC] inputs, transposed
  static constexpr uint32_t OFF_Y = OFF_X + uint32_t(D) * RPC * 4;     // [RPC][128] rotated slice
  static constexpr uint32_t OFF_M = OFF_Y + uint32_t(RPC) * kGroup * 4;  // [RPC] slice max |y|, [RPC] finite
  static constexpr uint32_t OFF_BAR = (OFF_M + 2 * RPC * 4 + 7) & ~7u;
  static constexpr uint32_t SMEM = OFF_BAR + 8 * NSTG;
  static_assert(RPC % 4 == 0, "rows per CTA must be a multiple of the warp count");
};

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_barrier() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t ld_cluster_u32(uint32_t saddr, uint32_t rank) {
  uint32_t remote, v;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(saddr), "r"(rank));
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(remote) : "memory");
  return v;
}

template <int D, int RPC>
__global__ void __launch_bounds__(kAppendThreads)
    kv_append_slices_kernel(const __grid_constant__ CUtensorMap tmRK, const __grid_constant__ CUtensorMap tmRV,
                            const AppendArgs a) {
  using C = SliceCfg<D, RPC>;
  extern __shared__ __align__(128) unsigned char sm[];
  float* Rs = reinterpret_cast<float*>(sm);                    // [NSTG][CH_ROWS][128]
  float* xs = reinterpret_cast<float*>(sm + C::OFF_X);         // [D][RPC]
  float* ys = reinterpret_cast<float*>(sm + C::OFF_Y);         // [RPC][128]
  uint32_t* ms = reinterpret_cast<uint32_t*>(sm + C::OFF_M);   // [RPC] max |y| bits, [RPC] finite
  const uint32_t bar0 = smem_u32(sm + C::OFF_BAR);

  pdl_wait();  // as in kv_append_rows_kernel
  pdl_trigger();
  const int role = blockIdx.y;
  const int q = int(cluster_rank());                  // quant group of this CTA
  const int64_t row0 = int64_t(blockIdx.x / C::SL) * RPC;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const CUtensorMap* tmR = role ? &tmRV : &tmRK;
  const int col0 = q * kGroup;

  // 1. R's column slice, one 64-row box per chunk (thread 0)
  auto issue_chunk = [&](int ch, int s) {
    mbar_arrive_expect_tx(bar0 + 8 * s, C::CH_BYTES);
    tma_load_2d(smem_u32(Rs) + s * C::CH_BYTES, tmR, col0, ch * C::CH_ROWS, bar0 + 8 * s);
  };
  if (tid == 0) {
    for (int s = 0; s < C::NSTG; ++s) mbar_init(bar0 + 8 * s, 1);
    mbar_fence_init();
  }
  __syncthreads();
  if (tid == 0)
    for (int s = 0; s < C::NSTG && s < C::NCH; ++s) issue_chunk(s, s);
  // inputs, 8 channels per load, stored transposed; rows past the end are zero
  for (int idx = tid; idx < RPC * (D / 8); idx += kAppendThreads) {
    const int r = idx / (D / 8), i0 = (idx % (D / 8)) * 8;
    const int64_t row = row0 + r;
    float v[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) v[e] = 0.f;
    if (row < a.rows) {
      if (a.in_fp32) {
        const float4* src = reinterpret_cast<const float4*>(static_cast<const float*>(role ? a.v_new : a.k_new) +
                                                            row * D + i0);
        const float4 u0 = src[0], u1 = src[1];
        v[0] = u0.x; v[1] = u0.y; v[2] = u0.z; v[3] = u0.w;
        v[4] = u1.x; v[5] = u1.y; v[6] = u1.z; v[7] = u1.w;
      } else {
        const uint4 u = *reinterpret_cast<const uint4*>(
            static_cast<const __nv_bfloat16*>(role ? a.v_new : a.k_new) + row * D + i0);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          v[2 * e] = __uint_as_float(w[e] << 16);
          v[2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
        }
      }
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) xs[(i0 + e) * RPC + r] = v[e];
  }
  __syncthreads();

  // 2. column col0 + tid of every row, fp32 FMAs in increasing input channel
  float acc[RPC];
#pragma unroll
  for (int r = 0; r < RPC; ++r) acc[r] = 0.f;
  bool ok = true;
  int ch = 0;
  for (; ch < C::NCH; ++ch) {
    const int s = ch % C::NSTG;
    const bool got = mbar_wait(bar0 + 8 * s, (ch / C::NSTG) & 1);
    if (__syncthreads_or(!got)) {
      ok = false;
      break;
    }
    const float* Rc = Rs + size_t(s) * C::CH_ROWS * kGroup;
#pragma unroll 4
    for (int kk = 0; kk < C::CH_ROWS; ++kk) {
      const int k = ch * C::CH_ROWS + kk;
      float xv[RPC];
#pragma unroll
      for (int r4 = 0; r4 < RPC / 4; ++r4) {
        const float4 x4 = *reinterpret_cast<const float4*>(xs + k * RPC + 4 * r4);
        xv[4 * r4 + 0] = x4.x;
        xv[4 * r4 + 1] = x4.y;
        xv[4 * r4 + 2] = x4.z;
        xv[4 * r4 + 3] = x4.w;
      }
      const float rv = Rc[kk * kGroup + tid];
#pragma unroll
      for (int r = 0; r < RPC; ++r) acc[r] = fmaf(xv[r], rv, acc[r]);
    }
    __syncthreads();  // every thread is done with stage s
    if (tid == 0 && ch + C::NSTG < C::NCH) issue_chunk(ch + C::NSTG, s);
  }
  if (!ok && tid == 0) {
    status_or(a.status, OSCAR_DEV_TIMEOUT);
    for (int c2 = ch; c2 < C::NCH && c2 < ch + C::NSTG; ++c2)
      (void)mbar_wait(bar0 + 8 * (c2 % C::NSTG), (c2 / C::NSTG) & 1);
  }
#pragma unroll
  for (int r = 0; r < RPC; ++r) ys[r * kGroup + tid] = acc[r];
  __syncthreads();

  // 3. this slice's max |y| and finiteness per row, then the row's over the cluster
  for (int r = warp; r < RPC; r += kAppendThreads / 32) {
    float amax = 0.f;
    bool finite = true;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float v = ys[r * kGroup + lane + 32 * e];
      finite &= isfinite(v);
      amax = fmaxf(amax, fabsf(v));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    finite = __all_sync(0xffffffffu, finite);
    if (lane == 0) {
      ms[r] = __float_as_uint(amax);
      ms[RPC + r] = finite ? 1u : 0u;
    }
  }
  cluster_barrier();
  float row_amax[RPC / 4];
  bool row_finite[RPC / 4];
#pragma unroll
  for (int i = 0; i < RPC / 4; ++i) {
    const int r = warp + 4 * i;
    float m = 0.f;
    bool f = true;
    if (lane < C::SL) {
      m = __uint_as_float(ld_cluster_u32(smem_u32(ms + r), uint32_t(lane)));
      f = ld_cluster_u32(smem_u32(ms + RPC + r), uint32_t(lane)) != 0u;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    row_amax[i] = m;
    row_finite[i] = __all_sync(0xffffffffu, f);
  }
  cluster_barrier();  // no CTA leaves while another reads its shared memory
  if (!ok) return;

  // 4. codec of this CTA's group, one warp per row
  const float ratio = role ? a.v_clip : a.k_clip;
  const Geom& g = a.g;
  uint8_t* role_base = a.layer_base + role * g.role_bytes;
#pragma unroll
  for (int i = 0; i < RPC / 4; ++i) {
    const int r = warp + 4 * i;
    const int64_t row = row0 + r;
    if (row >= a.rows) break;
    const float* y = ys + r * kGroup;
    float v[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) v[e] = y[lane + 32 * e];
    if (a.debug_rot) {
      float* dst = a.debug_rot + (row * 2 + role) * D + col0;
#pragma unroll
      for (int e = 0; e < 4; ++e) dst[lane + 32 * e] = v[e];
    }
    const int h = int(row % g.Hkv);
    const int64_t bt = row / g.Hkv;
    const int t = int(bt % a.n_new);
    const int b = int(bt / a.n_new);
    const int p = a.start_pos[b] + t;
    const int newlen = a.start_pos[b] + a.n_new;
    if (p < 0 || p >= g.cap) {
      if (lane == 0) status_or(a.status, OSCAR_DEV_OVER_CAPACITY);
      continue;
    }
    const int64_t bh = int64_t(b) * g.Hkv + h;
    if (!row_finite[i] && lane == 0) status_or(a.status, OSCAR_DEV_NONFINITE);
    const float tclip = __fmul_rn(ratio, row_amax[i]);

    if (role == 1 && g.vb) {  // K-only INT2: the V row is kept BF16 at its position
      __nv_bfloat16* dv = reinterpret_cast<__nv_bfloat16*>(role_base + (bh * g.cap + p) * (2 * D)) + col0;
#pragma unroll
      for (int e = 0; e < 4; ++e) dv[lane + 32 * e] = __float2bfloat16_rn(v[e]);
      continue;
    }
    const bool to_sink = p < g.S;
    const bool to_ring = g.W > 0 && p >= newlen - g.W;
    if (to_sink || to_ring) {
      __nv_bfloat16* d0 = reinterpret_cast<__nv_bfloat16*>(
          to_sink ? role_base + (bh * g.S + p) * (2 * D) : role_base + g.sink_bytes + (bh * g.W + (p % g.W)) * (2 * D));
      __nv_bfloat16* d1 = (to_sink && to_ring)
                              ? reinterpret_cast<__nv_bfloat16*>(role_base + g.sink_bytes + (bh * g.W + (p % g.W)) * (2 * D))
                              : nullptr;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const __nv_bfloat16 bv = __float2bfloat16_rn(v[e]);
        d0[col0 + lane + 32 * e] = bv;
        if (d1) d1[col0 + lane + 32 * e] = bv;
      }
    }
    if (to_sink) continue;

    float mn = INFINITY, mx = -INFINITY;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float x = fminf(fmaxf(v[e], -tclip), tclip);
      mn = fminf(mn, x);
      mx = fmaxf(mx, x);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    }
    const float s32 = __fdiv_rn(__fsub_rn(mx, mn), g.lm ? kLmSpan : 3.0f);
    const __half sh = __float2half_rn(s32);
    const __half zh = __float2half_rn(mn);
    const float sf = __half2float(sh), zf = __half2float(zh);
    const bool rng_ok = isfinite(sf) && isfinite(zf);
    if (!rng_ok && lane == 0) status_or(a.status, OSCAR_DEV_FP16_RANGE);
    const bool gok = rng_ok && sf != 0.f;
    const float inv = gok ? __frcp_rn(sf) : 0.f;

    // word w = lane / 4 of the group, slots 4 (lane % 4) .. + 3
    const int64_t irow = bh * g.ncap + (p - g.S);
    uint32_t* codes = reinterpret_cast<uint32_t*>(role_base + g.sink_bytes + g.ring_bytes + irow * (D / 4));
    uint32_t* sz = reinterpret_cast<uint32_t*>(role_base + g.sink_bytes + g.ring_bytes + g.codes_bytes) +
                   irow * (D / kGroup);
    const int wi = lane >> 2, part = lane & 3;
    uint32_t word = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int sl = part * 4 + k;
      const float x = fminf(fmaxf(y[slot_channel(role, wi, sl)], -tclip), tclip);
      const float yq = __fmul_rn(__fsub_rn(x, zf), inv);
      int c = g.lm ? lm_code(yq) : min(max(__float2int_rn(yq), 0), 3);
      c = gok ? c : 0;
      word |= uint32_t(c) << (2 * sl);
    }
    word |= __shfl_xor_sync(0xffffffffu, word, 1);
    word |= __shfl_xor_sync(0xffffffffu, word, 2);
    if (part == 0) codes[8 * q + wi] = word;
    if (lane == 0) sz[q] = pack_half2(sh, zh);
  }
}

template <int D, int RPC, bool HAD>
int launch_append_rows(const AppendArgs& a, cudaStream_t stream) {
  using C = RowsCfg<D, RPC>;
  constexpr uint32_t smem = HAD ? C::SMEM_HAD : C::SMEM;
  static int attr_set[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    if (cudaFuncSetAttribute(kv_append_rows_kernel<D, RPC, HAD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem) != cudaSuccess)
      return OSCAR_ERR_LAUNCH;
    attr_set[dev] = 1;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned((a.rows + RPC - 1) / RPC), 2, 1);
  cfg.blockDim = dim3(kAppendThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kv_append_rows_kernel<D, RPC, HAD>, a) == cudaSuccess ? OSCAR_OK
                                                                                       : OSCAR_ERR_LAUNCH;
}

}  // namespace

// 2-D tiled TMA map of a row-major float32 matrix (declared in internal.h)
bool encode_f32_tiles(CUtensorMap* m, const float* ptr, uint64_t rows, uint64_t cols, uint32_t box_cols,
                      uint32_t box_rows) {
  typedef CUresult (*EncodeFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                               const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                               CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
  static EncodeFn enc = nullptr;
  if (!enc) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      enc = reinterpret_cast<EncodeFn>(p);
  }
  if (!enc || rows == 0 || cols == 0) return false;
  const cuuint64_t dims[2] = {cuuint64_t(cols), cuuint64_t(rows)};
  const cuuint64_t strides[1] = {cuuint64_t(cols) * 4};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(ptr), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {

template <int D, int RPC>
int launch_append_slices(const AppendArgs& a, cudaStream_t stream) {
  using C = SliceCfg<D, RPC>;
  static int attr_set[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    if (cudaFuncSetAttribute(kv_append_slices_kernel<D, RPC>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::SMEM) != cudaSuccess)
      return OSCAR_ERR_LAUNCH;
    attr_set[dev] = 1;
  }
  const int64_t blocks = (a.rows + RPC - 1) / RPC;
  if (blocks * C::SL > (int64_t(1) << 31) - 1) return OSCAR_ERR_UNSUPPORTED;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(blocks * C::SL), 2, 1);
  cfg.blockDim = dim3(kAppendThreads, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C::SL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  CUtensorMap mk, mv;
  if (!encode_f32_tiles(&mk, a.R_K, D, D, kGroup, C::CH_ROWS) || !encode_f32_tiles(&mv, a.R_V, D, D, kGroup, C::CH_ROWS))
    return OSCAR_ERR_LAUNCH;
  return cudaLaunchKernelEx(&cfg, kv_append_slices_kernel<D, RPC>, mk, mv, a) == cudaSuccess ? OSCAR_OK
                                                                                            : OSCAR_ERR_LAUNCH;
}

// Row-parallel appends: at head_dim 256 / 512 and up to kSmallAppendRows rows
// per role (a decode step) a cluster of D / 128 CTAs, one per quant group, per
// RPC rows (decode-step append of 32 rows per role at head_dim 512: 37.5 ->
// 17.1 us); otherwise one CTA per RPC rows (larger K-only-INT2 or Lloyd-Max
// appends, where the sliced grid's per-CTA set-up costs more than the shared
// stream of R saves: 65,536 rows per role 3.3 vs 4.7 ms).
template <int D>
int launch_append_small(const AppendArgs& a, cudaStream_t stream) {
  if constexpr (D >= 256) {
    if (a.rows <= kSmallAppendRows)
      return a.rows > 512 ? launch_append_slices<D, 8>(a, stream) : launch_append_slices<D, 4>(a, stream);
  }
  return a.rows > 512 ? launch_append_rows<D, 8, false>(a, stream) : launch_append_rows<D, 4, false>(a, stream);
}

// the in-quant Hadamard reads no matrix, so every append takes the
// row-parallel kernel
template <int D>
int launch_append_hadamard(const AppendArgs& a, cudaStream_t stream) {
  return a.rows > 512 ? launch_append_rows<D, 8, true>(a, stream) : launch_append_rows<D, 4, true>(a, stream);
}

template <int D>
int launch_append_d(const AppendArgs& a, cudaStream_t stream) {
  using C = AppendCfg<D>;
  static int attr_set[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    if (cudaFuncSetAttribute(kv_append_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) !=
        cudaSuccess)
      return OSCAR_ERR_LAUNCH;
    attr_set[dev] = 1;
  }
  const dim3 grid(unsigned((a.rows + C::RPC - 1) / C::RPC), 2, 1);
  kv_append_kernel<D><<<grid, kAppendThreads, C::SMEM, stream>>>(a);
  return cudaGetLastError() == cudaSuccess ? OSCAR_OK : OSCAR_ERR_LAUNCH;
}

}  // namespace

int launch_append(const AppendArgs& a, cudaStream_t stream) {
  if (a.rows == 0) return OSCAR_OK;
  if (a.hadamard) {
    switch (a.g.D) {
      case 128: return launch_append_hadamard<128>(a, stream);
      case 256: return launch_append_hadamard<256>(a, stream);
      case 512: return launch_append_hadamard<512>(a, stream);
      default: return OSCAR_ERR_UNSUPPORTED;
    }
  }
  // K-only INT2 (V kept BF16) and Lloyd-Max levels are written by the
  // row-parallel kernel at every size
  if (a.rows <= kSmallAppendRows || a.g.vb || a.g.lm) {
    switch (a.g.D) {
      case 128: return launch_append_small<128>(a, stream);
      case 256: return launch_append_small<256>(a, stream);
      case 512: return launch_append_small<512>(a, stream);
      default: return OSCAR_ERR_UNSUPPORTED;
    }
  }
  if (a.g.D == 128 && !a.in_fp32 && a.rows < (int64_t(1) << 31)) return launch_append_tc(a, stream);
  switch (a.g.D) {
    case 128: return launch_append_d<128>(a, stream);
    case 256: return launch_append_d<256>(a, stream);
    case 512: return launch_append_d<512>(a, stream);
    default: return OSCAR_ERR_UNSUPPORTED;
  }
}

}  // namespace oscar
