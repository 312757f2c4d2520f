// kv_append on the 5th-generation tensor cores (head_dim 128, bf16 inputs).
//
// Same computation as kv_append.cu (rotate, clip, group-128 INT2 codes, BF16
// windows; see the Qwen3-4B model card, Run, and OSCAR-RotationZoo, How to use),
// organised as a GEMM [rows x 128] x [128 x 128] per role:
//
//   * R (float32) is split once per CTA into three bf16 matrices whose sum is R
//     exactly (8 + 8 + 8 mantissa bits); each bf16 product with a bf16 input is
//     exact, so the fp32 accumulation gives the rotation to float32 accuracy.
//     The pieces are written to shared memory transposed (N x K, K-major) in the
//     128-byte swizzled layout the MMA descriptors expect.
//   * A tiles of 128 rows are fetched with TMA tensor loads (cp.async.bulk.tensor,
//     SWIZZLE_128B) into a 4-stage ring by a loader warp of their own, which
//     refills a stage as soon as the MMAs reading it complete; it starts while
//     the other warps build R's pieces.
//   * One thread of the MMA warp issues 3 x 8 tcgen05.mma (M128 N128 K16,
//     kind::f16, bf16 operands, fp32 accumulate) per tile into one of four TMEM
//     accumulators and signals completion with tcgen05.commit.  It waits only
//     for its tile's data and accumulator: the tensor pipe, ~1 us per tile for
//     the three pieces, is what bounds this kernel, so no other wait may sit
//     between two tiles' MMAs.
//   * Sixteen epilogue warps in four groups (tile 4k + g goes to group g, with
//     accumulator g; four warps per SM sub-partition hide the codec's latency)
//     read their 32 TMEM lanes (one row per thread) with tcgen05.ld and run the
//     codec exactly as the CUDA-core kernel does, in two
//     passes: row min/max (which give max|x| and, clamping being monotone, the
//     clipped group min/max), then codes and BF16 copies.
//
// Every wait is bounded; on a timeout the kernel flags OSCAR_DEV_TIMEOUT, stops
// issuing work, waits (bounded) for its own copies and MMAs and frees TMEM.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>

#include "internal.h"

namespace oscar {
namespace {

constexpr int kD = 128;
constexpr int kTileRows = 128;
constexpr int kEpiWarps = 16;                // four groups of four: tiles 4k + group
constexpr int kMmaWarp = kEpiWarps;          // one thread issues the MMAs
constexpr int kLoadWarp = kEpiWarps + 1;     // one thread issues the TMA loads
constexpr int kThreadsTc = (kEpiWarps + 2) * 32;
constexpr int kComputeThreads = (kEpiWarps + 1) * 32;  // every warp but the loader
constexpr uint32_t kKBlockBytes = kTileRows * 128;  // 128 rows x 64 bf16 (128 B), swizzled
constexpr uint32_t kOperandBytes = 2 * kKBlockBytes; // K = 128 -> two K-blocks
constexpr uint32_t kOffB = 0;                          // 3 pieces of R^T
constexpr int kStagesA = 4;                            // A ring depth
constexpr uint32_t kOffA = 3 * kOperandBytes;          // kStagesA stages of A
constexpr uint32_t kOffBar = kOffA + kStagesA * kOperandBytes;
constexpr uint32_t kSmemTc = kOffBar + 128 + 1024;     // + alignment slack
constexpr uint32_t kTmemCols = 512;                    // four 128-column fp32 accumulators
constexpr int kSposCache = 256;                        // start positions staged in shared memory

// UMMA shared-memory descriptor: K-major, 128-byte swizzle, 8-row groups 1024 B apart.
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= uint64_t((saddr >> 4) & 0x3FFF);        // start address
  d |= uint64_t(1) << 16;                       // leading byte offset (unused for swizzled K-major)
  d |= uint64_t(1024 >> 4) << 32;               // stride byte offset
  d |= uint64_t(1) << 46;                       // descriptor version
  d |= uint64_t(2) << 61;                       // 128-byte swizzle
  return d;
}

// Instruction descriptor: kind::f16, bf16 A/B, fp32 D, K-major A and B, M=128, N=128.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(kD >> 3) << 17) |
                            (uint32_t(kTileRows >> 4) << 24);

__device__ __forceinline__ void umma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(
          tmem_d),
      "l"(adesc), "l"(bdesc), "r"(kIdesc), "r"(acc)
      : "memory");
}

__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

// tcgen05.ld of 32 consecutive fp32 columns of the thread's TMEM lane, without
// the wait; tmem_wait32 waits for all of the thread's loads and carries the
// registers, so nothing reads them before they have landed.
__device__ __forceinline__ void tmem_ld32_start(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
               : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait32(uint32_t (&r)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
               :
               : "memory");
}

// 64 consecutive fp32 columns of the thread's TMEM lane; the wait carries the
// registers so nothing reads them before the load has landed.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float (&v)[64]) {
  uint32_t r[64];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31]), "+r"(r[32]), "+r"(r[33]), "+r"(r[34]), "+r"(r[35]), "+r"(r[36]), "+r"(r[37]), "+r"(r[38]), "+r"(r[39]), "+r"(r[40]), "+r"(r[41]), "+r"(r[42]), "+r"(r[43]), "+r"(r[44]), "+r"(r[45]), "+r"(r[46]), "+r"(r[47]), "+r"(r[48]), "+r"(r[49]), "+r"(r[50]), "+r"(r[51]), "+r"(r[52]), "+r"(r[53]), "+r"(r[54]), "+r"(r[55]), "+r"(r[56]), "+r"(r[57]), "+r"(r[58]), "+r"(r[59]), "+r"(r[60]), "+r"(r[61]), "+r"(r[62]), "+r"(r[63])
               :
               : "memory");
#pragma unroll
  for (int j = 0; j < 64; ++j) v[j] = __uint_as_float(r[j]);
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Byte offset of element (row, k) of a K-major, 128-byte-swizzled operand with
// 128 rows and K = 128 (two 64-element K-blocks).
__device__ __forceinline__ uint32_t sw128_offset(int row, int k) {
  const int kb = k >> 6, kin = k & 63;
  const int chunk = (kin >> 3) ^ (row & 7);
  return uint32_t(kb) * kKBlockBytes + uint32_t(row) * 128 + uint32_t(chunk) * 16 + uint32_t(kin & 7) * 2;
}

__global__ void __launch_bounds__(kThreadsTc, 1)
    kv_append_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                        const AppendArgs a) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  __shared__ int spos[kSposCache];  // start positions of the first kSposCache sequences
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  const uint32_t sB = base + kOffB, sA = base + kOffA;
  const uint32_t bar0 = base + kOffBar;
  auto full_a = [&](int s) { return bar0 + 8u * s; };          // s < kStagesA
  auto empty_a = [&](int s) { return bar0 + 32u + 8u * s; };    // s < kStagesA
  auto acc_full = [&](int s) { return bar0 + 64u + 8u * s; };   // s < 4
  auto acc_empty = [&](int s) { return bar0 + 96u + 8u * s; };  // s < 4

  pdl_trigger();  // a dependent kernel may be scheduled now; it waits for our completion itself
  const int role = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float* __restrict__ R = role ? a.R_V : a.R_K;
  const CUtensorMap* tmap = role ? &tmV : &tmK;
  const int64_t ntiles = (a.rows + kTileRows - 1) / kTileRows;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int s = 0; s < kStagesA; ++s) {
      mbar_init(full_a(s), 1);
      mbar_init(empty_a(s), 1);
    }
    for (int s = 0; s < 4; ++s) {
      mbar_init(acc_full(s), 1);
      mbar_init(acc_empty(s), kEpiWarps / 4);  // the four warps of the group that drains it
    }
    mbar_fence_init();
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();  // barriers initialised: the loader starts while the others build B

  // this CTA's tiles j = 0, 1, ...: tile blockIdx.x + j * gridDim.x, A stage j % kStagesA
  const int64_t my_tiles = blockIdx.x < ntiles ? (ntiles - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
  if (warp == kLoadWarp) {
    // ------------------------------ TMA loader -------------------------------
    // Refills a stage as soon as the MMAs of the tile in it have completed, up
    // to kStagesA tiles ahead of the MMA issuer.
    if (lane == 0) {
      int loaded = 0;
      bool ok = true;
      for (int j = 0; j < my_tiles; ++j) {
        const int s = j % kStagesA;
        if (j >= kStagesA) ok = mbar_wait(empty_a(s), ((j / kStagesA) & 1) ^ 1);
        if (!ok || *((volatile int*)&abort_flag)) break;
        const int64_t tile = blockIdx.x + int64_t(j) * gridDim.x;
        mbar_arrive_expect_tx(full_a(s), kOperandBytes);
        const uint32_t dst = sA + s * kOperandBytes;
        tma_load_2d(dst, tmap, 0, int(tile * kTileRows), full_a(s));
        tma_load_2d(dst + kKBlockBytes, tmap, 64, int(tile * kTileRows), full_a(s));
        ++loaded;
      }
      if (!ok) {
        abort_flag = 1;
        status_or(a.status, OSCAR_DEV_TIMEOUT);
      }
      // every copy issued lands before the CTA exits (tiles before the last
      // kStagesA were consumed: their stages were refilled)
      for (int j = (loaded > kStagesA ? loaded - kStagesA : 0); j < loaded; ++j)
        (void)mbar_wait(full_a(j % kStagesA), (j / kStagesA) & 1);
    }
    return;  // the barriers below are named ones that leave the loader out
  }
  // B operand: piece p holds B_p[n][k] with R[k][n] = B_0 + B_1 + B_2 (bf16).
  // Each thread builds one 16-byte chunk of each piece: 8 consecutive k of row
  // n.  Consecutive threads take consecutive n, so every load of R is a
  // coalesced row segment and the chunk stores of a warp spread over all banks
  // (the 128-byte swizzle puts rows n and n + 1 .. n + 7 in different chunks).
  for (int cidx = threadIdx.x; cidx < kD * (kD / 8); cidx += kComputeThreads) {
    const int n = cidx % kD, k0 = (cidx / kD) * 8;
    uint32_t ph[4], pm[4], pl[4];
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
      uint32_t p0[3], p1[3];
      split3_bf16(__ldg(R + (k0 + e) * kD + n), p0);
      split3_bf16(__ldg(R + (k0 + e + 1) * kD + n), p1);
      ph[e / 2] = p0[0] | (p1[0] << 16);
      pm[e / 2] = p0[1] | (p1[1] << 16);
      pl[e / 2] = p0[2] | (p1[2] << 16);
    }
    const uint32_t off = sw128_offset(n, k0);
    *reinterpret_cast<uint4*>(smem + kOffB + 0 * kOperandBytes + off) = make_uint4(ph[0], ph[1], ph[2], ph[3]);
    *reinterpret_cast<uint4*>(smem + kOffB + 1 * kOperandBytes + off) = make_uint4(pm[0], pm[1], pm[2], pm[3]);
    *reinterpret_cast<uint4*>(smem + kOffB + 2 * kOperandBytes + off) = make_uint4(pl[0], pl[1], pl[2], pl[3]);
  }
  for (int i = threadIdx.x; i < a.g.B && i < kSposCache; i += kComputeThreads) spos[i] = a.start_pos[i];
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // make generic smem writes visible to the MMA
  tc_fence_before();
  asm volatile("bar.sync 1, %0;" ::"r"(kComputeThreads) : "memory");  // B and spos ready (not the loader)
  tc_fence_after();
  const uint32_t tmem = tmem_slot;

  if (warp == kMmaWarp) {
    // ------------------------------ MMA issuer -------------------------------
    if (lane == 0) {
      bool ok = true;
      int it = 0;
      for (; it < my_tiles; ++it) {
        const int s = it % kStagesA;  // A stage
        const uint32_t ph = (it / kStagesA) & 1;
        const int sa = it & 3;  // TMEM accumulator
        const uint32_t pa = (it >> 2) & 1;
        if (*((volatile int*)&abort_flag)) ok = false;
        if (ok) ok = mbar_wait(full_a(s), ph);
        if (ok && it >= 4) ok = mbar_wait(acc_empty(sa), pa ^ 1);
        if (!ok) break;
        tc_fence_after();
        const uint32_t dcol = tmem + uint32_t(sa) * kD;
        const uint32_t a_base = sA + s * kOperandBytes;
#pragma unroll
        for (int p = 0; p < 3; ++p) {
#pragma unroll
          for (int k = 0; k < kD / 16; ++k) {
            const uint32_t koff = uint32_t(k >> 2) * kKBlockBytes + uint32_t(k & 3) * 32;
            umma_bf16(dcol, umma_desc_sw128(a_base + koff), umma_desc_sw128(sB + p * kOperandBytes + koff),
                      (p | k) != 0);
          }
        }
        umma_commit(acc_full(sa));
        umma_commit(empty_a(s));
      }
      if (!ok) {
        abort_flag = 1;
        status_or(a.status, OSCAR_DEV_TIMEOUT);
      }
      // drain: the last (up to four) commits must have landed before TMEM is freed
      for (int j = (it >= 4 ? it - 4 : 0); j < it; ++j) mbar_wait(acc_full(j & 3), (j >> 2) & 1);
    }
  } else {
    // ------------------------------- epilogue --------------------------------
    const Geom& g = a.g;
    const float ratio = role ? a.v_clip : a.k_clip;
    uint8_t* role_base = a.layer_base + role * g.role_bytes;
    const int grp = warp >> 2, quarter = warp & 3;  // tile group (= accumulator), TMEM lane quarter
    int it = grp;
    for (int64_t tile = blockIdx.x + int64_t(grp) * gridDim.x; tile < ntiles;
         tile += 4 * int64_t(gridDim.x), it += 4) {
      const int s = it & 3;
      int ok = 1;
      if (lane == 0) ok = mbar_wait(acc_full(s), (it >> 2) & 1);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) {
        if (lane == 0) { abort_flag = 1; status_or(a.status, OSCAR_DEV_TIMEOUT); }
        break;
      }
      tc_fence_after();
      const uint32_t taddr = tmem + (uint32_t(32 * quarter) << 16) + uint32_t(s) * kD;
      const int64_t row = tile * kTileRows + 32 * quarter + lane;
      const bool valid = row < a.rows;

      // pass 1: raw row min / max (NaN-propagating, so a NaN row shows as non-finite).
      // The loops over the four 32-column chunks stay rolled: sixteen warps run
      // this code and it must fit the instruction cache.
      // Two 64-column loads, each reduced in two independent chains.
      float rmn = INFINITY, rmx = -INFINITY;
      {
        float rmn1 = INFINITY, rmx1 = -INFINITY;
#pragma unroll 1
        for (int c = 0; c < 2; ++c) {
          float w[64];
          tmem_ld64(taddr + 64 * c, w);
#pragma unroll
          for (int j = 0; j < 64; j += 4) {
            rmn = fmin3_nan(rmn, w[j], w[j + 1]);
            rmx = fmax3_nan(rmx, w[j], w[j + 1]);
            rmn1 = fmin3_nan(rmn1, w[j + 2], w[j + 3]);
            rmx1 = fmax3_nan(rmx1, w[j + 2], w[j + 3]);
          }
        }
        rmn = fmin_nan(rmn, rmn1);
        rmx = fmax_nan(rmx, rmx1);
      }
      const bool finite = isfinite(rmn) && isfinite(rmx);
      const float amax = fmaxf(fabsf(rmn), fabsf(rmx));          // max_j |r_j|
      const float tclip = __fmul_rn(ratio, amax);
      const float mn = fminf(fmaxf(rmn, -tclip), tclip);           // min_j clamp(r_j)
      const float mx = fminf(fmaxf(rmx, -tclip), tclip);           // max_j clamp(r_j)
      const float s32 = __fdiv_rn(__fsub_rn(mx, mn), 3.0f);
      const __half sh = __float2half_rn(s32);
      const __half zh = __float2half_rn(mn);
      const float sf = __half2float(sh), zf = __half2float(zh);
      const bool rng_ok = isfinite(sf) && isfinite(zf);
      const bool qok = rng_ok && sf != 0.f;
      const float inv = qok ? __frcp_rn(sf) : 0.f;
      const uint64_t zz = splat_x2(zf), ii = splat_x2(inv);

      int b = 0, p = -1, newlen = 0;
      int64_t bh = 0;
      if (valid) {
        // row = (b n_new + t) Hkv + h, below 2^31 on this path
        const uint32_t r32 = uint32_t(row);
        const uint32_t bt = fastdiv(r32, a.div_hkv);
        const int h = int(r32 - bt * uint32_t(g.Hkv));
        const uint32_t bq = fastdiv(bt, a.div_n_new);
        const int t = int(bt - bq * uint32_t(a.n_new));
        b = int(bq);
        const int sp = b < kSposCache ? spos[b] : a.start_pos[b];
        p = sp + t;
        newlen = sp + a.n_new;
        bh = int64_t(b) * g.Hkv + h;
        if (!finite) status_or(a.status, OSCAR_DEV_NONFINITE);
        if (!rng_ok) status_or(a.status, OSCAR_DEV_FP16_RANGE);
        if (p < 0 || p >= g.cap) status_or(a.status, OSCAR_DEV_OVER_CAPACITY);
      }
      const bool in_cache = valid && p >= 0 && p < g.cap;
      const bool to_sink = in_cache && p < g.S;
      const bool to_ring = in_cache && g.W > 0 && p >= newlen - g.W;
      uint4* sink4 = to_sink ? reinterpret_cast<uint4*>(role_base + (bh * g.S + p) * (2 * kD)) : nullptr;
      uint4* ring4 =
          to_ring ? reinterpret_cast<uint4*>(role_base + g.sink_bytes + (bh * g.W + (p % g.W)) * (2 * kD)) : nullptr;
      float4* dbg = (valid && a.debug_rot) ? reinterpret_cast<float4*>(a.debug_rot + (row * 2 + role) * kD) : nullptr;

      // pass 2: codes, BF16 windows, debug rows
      uint32_t words[8];
#pragma unroll
      for (int w = 0; w < 8; ++w) words[w] = 0;
      // one 32-column chunk c of the row, raw TMEM words in r
      auto chunk = [&](const uint32_t (&r)[32], const int c) {
        float v[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
        if (dbg) {
#pragma unroll
          for (int j = 0; j < 32; j += 4) dbg[(32 * c + j) / 4] = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
        }
        if (sink4 || ring4) {
#pragma unroll
          for (int j = 0; j < 32; j += 8) {
            uint4 q;
            q.x = pack_bf162(__float2bfloat16_rn(v[j + 0]), __float2bfloat16_rn(v[j + 1]));
            q.y = pack_bf162(__float2bfloat16_rn(v[j + 2]), __float2bfloat16_rn(v[j + 3]));
            q.z = pack_bf162(__float2bfloat16_rn(v[j + 4]), __float2bfloat16_rn(v[j + 5]));
            q.w = pack_bf162(__float2bfloat16_rn(v[j + 6]), __float2bfloat16_rn(v[j + 7]));
            if (sink4) sink4[(32 * c + j) / 8] = q;
            if (ring4) ring4[(32 * c + j) / 8] = q;
          }
        }
        // code = clamp(rint((clamp(r, -t, t) - z) * inv), 0, 3) as the codec
        // defines it, evaluated without the clamp of r and without a qok
        // select: (1) where r > t, the group's max was clipped to t, so
        // (t - z) * inv rounds to 3 and, every step being monotone, r gives a
        // code >= 3 as well; symmetrically below -t, and a group with no
        // clipped value has no r beyond t; (2) inv = 0 when !qok, so the
        // product is 0 (or NaN for a non-finite zero, which cvt.rni turns into 0).
        // Channels go in pairs through one packed subtract and multiply.
        float cf[32];
#pragma unroll
        for (int j = 0; j < 32; j += 2) sub_mul_x2(v[j], v[j + 1], zz, ii, cf[j], cf[j + 1]);
        auto code_of = [&](int j) {
          return min(__float2uint_rn(cf[j]), 3u);  // the conversion saturates below 0
        };
        // the role is uniform per CTA: one loop per code layout.  Channel
        // d = 32 c + j; the chunk's codes are gathered with shifts that do not
        // depend on c, then moved into place.  Codes occupy disjoint bit
        // pairs, so they are combined with additions (shift-and-add is one
        // instruction).
        if (role == 0) {
          // K: word 2 (e >> 1) + (c >> 1), bit 8 (c & 1) + 4 (j >> 4) + 2 hh + 16 (e & 1)
          // with e = j & 7, hh = (j >> 3) & 1 (the header's K layout for d)
          uint32_t wl[4] = {0u, 0u, 0u, 0u};
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int e = j & 7, hh = (j >> 3) & 1;
            wl[e >> 1] += code_of(j) << (4 * (j >> 4) + 2 * hh + 16 * (e & 1));
          }
          const int sh = 8 * (c & 1);
          const bool hi = (c >> 1) != 0;
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            const uint32_t x = wl[m] << sh;
            words[2 * m] |= hi ? 0u : x;
            words[2 * m + 1] |= hi ? x : 0u;
          }
        } else {
          // V: word d & 7 = j & 7, bit 2 (d >> 3) = 8 c + 2 (j >> 3)
          uint32_t wl[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
#pragma unroll
          for (int j = 0; j < 32; ++j) wl[j & 7] += code_of(j) << (2 * (j >> 3));
#pragma unroll
          for (int m = 0; m < 8; ++m) words[m] |= wl[m] << (8 * c);
        }
      };
      uint32_t ra[32];
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        tmem_ld32_start(taddr + 32 * c, ra);
        tmem_wait32(ra);
        chunk(ra, c);
      }
      if (in_cache && p >= g.S) {
        const int64_t irow = bh * g.ncap + (p - g.S);
        uint4* c4 = reinterpret_cast<uint4*>(role_base + g.sink_bytes + g.ring_bytes + irow * (kD / 4));
        c4[0] = make_uint4(words[0], words[1], words[2], words[3]);
        c4[1] = make_uint4(words[4], words[5], words[6], words[7]);
        reinterpret_cast<uint32_t*>(role_base + g.sink_bytes + g.ring_bytes + g.codes_bytes)[irow] =
            pack_half2(sh, zh);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acc_empty(s));
    }
  }
  tc_fence_before();
  asm volatile("bar.sync 1, %0;" ::"r"(kComputeThreads) : "memory");  // every MMA and TMEM load is done
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_slot), "r"(kTmemCols)
                 : "memory");
  }
}

}  // namespace

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

bool encode_rows_bf16(CUtensorMap* m, const void* ptr, uint64_t rows, uint32_t cols, uint32_t box_cols,
                      uint32_t box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc || rows == 0) return false;
  const cuuint64_t dims[2] = {cuuint64_t(cols), cuuint64_t(rows)};
  const cuuint64_t strides[1] = {cuuint64_t(cols) * 2};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_code_rows(CUtensorMap* m, const void* ptr, uint64_t rows, uint32_t rowb, uint32_t box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc || rows == 0) return false;
  const CUtensorMapSwizzle sw = rowb == 32   ? CU_TENSOR_MAP_SWIZZLE_32B
                                : rowb == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                             : CU_TENSOR_MAP_SWIZZLE_128B;
  if (rowb != 32 && rowb != 64 && rowb != 128) return false;
  const cuuint64_t dims[2] = {cuuint64_t(rowb), cuuint64_t(rows)};
  const cuuint64_t strides[1] = {cuuint64_t(rowb)};
  const cuuint32_t box[2] = {rowb, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {

bool make_rows_map(CUtensorMap* m, const void* ptr, int64_t rows) {
  return encode_rows_bf16(m, ptr, uint64_t(rows), kD, 64, kTileRows);
}

}  // namespace

int launch_append_tc(const AppendArgs& a, cudaStream_t stream) {
  static int attr_set[64] = {0};
  static int sms[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev >= 64) return OSCAR_ERR_LAUNCH;
  if (!attr_set[dev]) {
    if (cudaFuncSetAttribute(kv_append_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemTc) !=
            cudaSuccess ||
        cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return OSCAR_ERR_LAUNCH;
    attr_set[dev] = 1;
  }
  if (a.rows >= (int64_t(1) << 31)) return OSCAR_ERR_LAUNCH;  // 32-bit row indices and TMA coordinates
  CUtensorMap mk, mv;
  if (!make_rows_map(&mk, a.k_new, a.rows) || !make_rows_map(&mv, a.v_new, a.rows)) return OSCAR_ERR_LAUNCH;
  const int64_t ntiles = (a.rows + kTileRows - 1) / kTileRows;
  const int per_role = int(std::min<int64_t>(ntiles, std::max(1, sms[dev] / 2)));
  AppendArgs ka = a;
  ka.div_hkv = fastdiv_make(uint32_t(a.g.Hkv));
  ka.div_n_new = fastdiv_make(uint32_t(a.n_new));
  kv_append_tc_kernel<<<dim3(per_role, 2, 1), kThreadsTc, kSmemTc, stream>>>(mk, mv, ka);
  return cudaGetLastError() == cudaSuccess ? OSCAR_OK : OSCAR_ERR_LAUNCH;
}

}  // namespace oscar
