// kv_append: rotate new K/V rows by the layer's orthogonal matrix, clip each
// row, quantise groups of 128 channels to 2-bit codes with fp16 scale/zero and
// write the BF16 sink / recent-window copies.
//
// Source: "OSCAR-LLAMACPP-Qwen3-4B-Thinking-2507-INT2-KV" model card (Files
// note: post-RoPE orthogonal transform on K and V; Run: per-row clip ratio,
// high-precision sink/recent tokens) and "OSCAR-RotationZoo" (Available
// rotations: group 128 along head_dim; How to use: K/V clip 0.96/0.92).
//
// One CTA of 128 threads handles RPC = 128*128/D rows of one role (K or V):
//   1. stage the input rows in shared memory as float32;
//   2. rotate: each row's D outputs are split over 128/RPC threads, each
//      accumulating 32 columns at a time with fp32 FMAs (R is read through the
//      L1 as warp-wide broadcasts);
//   3. quantise: one thread per row, the row held in padded shared memory.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"

namespace oscar {
namespace {

constexpr int kAppendThreads = 128;

template <int D>
struct AppendCfg {
  static constexpr int RPC = kAppendThreads * 128 / D;  // rows per CTA
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
  if (a.g.D == 128 && !a.in_fp32) return launch_append_tc(a, stream);
  switch (a.g.D) {
    case 128: return launch_append_d<128>(a, stream);
    case 256: return launch_append_d<256>(a, stream);
    case 512: return launch_append_d<512>(a, stream);
    default: return OSCAR_ERR_UNSUPPORTED;
  }
}

}  // namespace oscar
