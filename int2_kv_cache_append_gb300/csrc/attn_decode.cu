// attn_decode: one decode step of attention over the mixed INT2 / BF16 cache.
//
// Source: hysenlabs article on FutureMLS-Lab/OSCAR (How the offline rotation
// is fit: a fused mixed-precision flash attention over the INT2 + BF16 layout,
// no dequantise-then-attend pass); "OSCAR-LLAMACPP-Gemma-4-12B-it-INT2-KV"
// card (Folders: the rotation applies to Q/K and V); "OSCAR-RotationZoo" (How
// to use: V rotation absorbed into the output).
//
// Two kernels per call:
//   qrot   q' = q R_K * sm_scale * log2(e) (float32) and per-group sums of q'.
//   split  grid (splits, Hkv, B).  Four consumer warps and one producer warp.
//          The producer streams 64-token INT2 blocks (codes + scale/zero) and
//          16-token BF16 blocks (sink, ring) into a shared-memory ring with
//          cp.async.bulk + mbarriers.  Consumers compute scores and P.V with
//          mma.sync m16n8k16 in "swap-AB" form: tokens (QK) or channels (PV)
//          on the M side, query heads on N, with each head's hi and lo fp16
//          (bf16 for BF16 blocks) split in adjacent columns so that the
//          products keep ~22 bits.  INT2 codes are unpacked straight into
//          A fragments (exact small integers); per-token scale/zero are
//          applied algebraically:
//            s_t = scale_t * (q'.c_t) + zero_t * sum(q'),
//            o  += (p_t * scale_t) . c_t  and  zeta += p_t * zero_t.
//          Online softmax in log2 units; teams of D/128 warps split the
//          channels of a block by quant group and exchange partial scores.
//          Each CTA writes one partial (m, l, o') per head; the last CTA of a
//          (b, kv head) to finish (an atomic ticket, never a wait) merges the
//          splits by log-sum-exp, applies o = o' R_V^T (skipped when absorbed)
//          and stores bf16/fp32 output and lse.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <cstring>

#include "internal.h"

namespace oscar {
namespace {

constexpr int kNCW = 4;                    // warps per CTA (each team issues its own copies)
constexpr int kThreads = kNCW * 32;
constexpr int kI2Tok = 128;                // tokens per INT2 block (one set of bulk copies)
constexpr int kSub = 64;                   // tokens per INT2 compute sub-block
constexpr int kBfTok = 16;                 // tokens per BF16 block

template <int D, int NQT>
struct DecCfg {
  static constexpr int Dg = D / kGroup;
  static constexpr int TS = Dg;              // warps per team (one quant group each)
  static constexpr int NTEAMS = kNCW / TS;
  static constexpr int ROWB = D / 4;         // code bytes per token
  static constexpr int BOXES = D / 64;       // 16-row x 64-column TMA boxes per BF16 matrix
  static constexpr int BOX_BYTES = kBfTok * 128;
  static constexpr int I2_BYTES = kI2Tok * (2 * ROWB + 2 * Dg * 4);
  static constexpr int BF_BYTES = 2 * BOXES * BOX_BYTES;
  static constexpr int STAGE = ((I2_BYTES > BF_BYTES ? I2_BYTES : BF_BYTES) + 1023) / 1024 * 1024;
  // Each team owns NSTW private stages: it issues the bulk copies of its own
  // blocks into them and consumes them in order, so a stage's barrier phases
  // are produced and awaited by one team only.
  static constexpr int NST = D == 128 ? 8 : (D == 256 ? 6 : 4);
  static_assert(NST % NTEAMS == 0, "every stage must belong to one team");
  static constexpr int NSTW = NST / NTEAMS;
  static constexpr int HEADS = 4 * NQT;      // head slots per (b, kv head)
  // shared memory carve-up (bytes)
  static constexpr int OFF_STAGE = 0;
  static constexpr int OFF_QBF = OFF_STAGE + NST * STAGE;           // bf16 q fragments per warp
  static constexpr int NQB = 2 * NQT;       // bf16 n-tiles: (hi, mid) and (lo, -) per 4 heads
  static constexpr int QBF_BYTES = TS * 8 * NQB * 32 * 8;  // one copy per channel group, shared by teams
  static constexpr int OFF_XCH = OFF_QBF + QBF_BYTES;               // team score exchange
  static constexpr int XCH_BYTES = TS > 1 ? NTEAMS * 2 * TS * kSub * HEADS * 4 : 0;
  static constexpr int OFF_PART = OFF_XCH + XCH_BYTES;              // team partials
  // team partials [team][head][D + 2]; reused by the merging CTA for o' [head][D],
  // max/sum [2][head] and split weights [head][OSCAR_KV_MAX_SPLITS]
  static constexpr int PART_A = NTEAMS * HEADS * (D + 2);
  static constexpr int PART_B = HEADS * (D + 2 + OSCAR_KV_MAX_SPLITS);
  static constexpr int PART_BYTES = (PART_A > PART_B ? PART_A : PART_B) * 4;
  static constexpr int OFF_BAR = OFF_PART + PART_BYTES;
  static constexpr int SMEM = OFF_BAR + (NST + 1) * 8 + 16 + 1024;  // + slack to align the base to 1 KB
};

// Per-(b, kv head) region sizes and the block list
struct Regions {
  int T, n_sink, tq, n_int, n_ring;
  int ra, rlen1, nrb1;  // ring: first slot, positions before the slot wrap, their blocks
  int nsb, nib, nrb;
  int64_t cbf, ci2;
};

__device__ __forceinline__ Regions make_regions(int T, int S, int W, int D) {
  Regions r;
  r.T = T;
  if (T <= S) {
    r.n_sink = T; r.tq = T; r.n_int = 0; r.n_ring = 0;
  } else {
    r.n_sink = S;
    r.tq = max(S, T - W);
    r.n_int = r.tq - S;
    r.n_ring = T - r.tq;
  }
  r.nsb = (r.n_sink + kBfTok - 1) / kBfTok;
  r.nib = (r.n_int + kI2Tok - 1) / kI2Tok;
  // ring positions [tq, T) sit in slots p mod W: cut them where the slots wrap
  // so that every block reads consecutive slots
  r.ra = r.n_ring > 0 ? r.tq % W : 0;
  r.rlen1 = r.n_ring > 0 ? min(r.n_ring, W - r.ra) : 0;
  r.nrb1 = (r.rlen1 + kBfTok - 1) / kBfTok;
  r.nrb = r.nrb1 + (r.n_ring - r.rlen1 + kBfTok - 1) / kBfTok;
  r.cbf = int64_t(2) * kBfTok * 2 * D;
  r.ci2 = int64_t(2) * kI2Tok * (D / 4 + 4 * (D / kGroup));
  return r;
}

// Smallest block index whose starting cost is >= x.
__device__ __forceinline__ int first_block_at(const Regions& r, int64_t x) {
  const int64_t c0 = r.nsb * r.cbf, c1 = c0 + r.nib * r.ci2;
  if (x <= 0) return 0;
  if (x <= c0) return int((x + r.cbf - 1) / r.cbf);
  if (x <= c1) return r.nsb + int((x - c0 + r.ci2 - 1) / r.ci2);
  const int k = r.nsb + r.nib + int((x - c1 + r.cbf - 1) / r.cbf);
  return min(k, r.nsb + r.nib + r.nrb);
}

struct Blk {
  int type;   // 0 sink, 1 int2, 2 ring
  int first;  // sink: first position; int2: first row (position - S); ring: first slot
  int count;
};

__device__ __forceinline__ Blk block_at(const Regions& r, int k) {
  Blk b;
  if (k < r.nsb) {
    b.type = 0; b.first = k * kBfTok; b.count = min(kBfTok, r.n_sink - b.first);
  } else if (k < r.nsb + r.nib) {
    b.type = 1; b.first = (k - r.nsb) * kI2Tok; b.count = min(kI2Tok, r.n_int - b.first);
  } else {
    const int kr = k - r.nsb - r.nib;
    b.type = 2;
    if (kr < r.nrb1) {
      b.first = r.ra + kr * kBfTok;
      b.count = min(kBfTok, r.rlen1 - kr * kBfTok);
    } else {
      b.first = (kr - r.nrb1) * kBfTok;
      b.count = min(kBfTok, r.n_ring - r.rlen1 - b.first);
    }
  }
  return b;
}

// AND of `v` over the `n` threads meeting at named barrier `id`.
__device__ __forceinline__ int team_all(int v, int id, int n) {
  int r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.s32 q, %1, 0;\n bar.red.and.pred p, %2, %3, q;\n selp.s32 %0, 1, 0, p;\n}\n"
      : "=r"(r)
      : "r"(v), "r"(id), "r"(n)
      : "memory");
  return r;
}

__device__ __forceinline__ int clamp_seq_len(const DecodeArgs& a, int b) {
  int T = a.seq_lens[b];
  if (T > a.g.cap) T = a.g.cap;
  if (T < 0) T = 0;
  return T;
}

// ---------------------------------------------------------------------------
// qrot: q' = q R_K * qscale and per-group sums for the G query heads of one
// (b, kv head) and one 128-column chunk of q'; the chunk-0 CTA also zeroes
// that unit's merge ticket.  512 threads = 4 slices of the contraction index
// x 128 output columns, so each thread has at most D/4 loads of R_K, issued
// 32 at a time.  Launched with PDL: it waits for the preceding kernel before
// reading anything (q may be produced right before this call) and then at
// once lets the split kernel launch, whose CTAs start their cache copies
// while this kernel computes; the split kernel reads q' only after its own
// wait for this grid's completion.
// ---------------------------------------------------------------------------
constexpr int kQrotThreads = 512;

template <int D>
__global__ void __launch_bounds__(kQrotThreads) qrot_kernel(const DecodeArgs a) {
  constexpr int KP = kQrotThreads / 128;  // slices of the contraction index
  constexpr int KC = D / KP;              // contraction indices per slice
  __shared__ float qs[8][D];
  __shared__ float part[KP - 1][8][128];
  __shared__ float red[8][4];
  const int bh = blockIdx.x;  // b * Hkv + h
  const int chunk = blockIdx.y;
  const int G = a.g.G;
  const int c = threadIdx.x & 127, kp = threadIdx.x >> 7;
  const int col = chunk * 128 + c;
  const int64_t q0 = int64_t(bh) * G * D;  // first query head of this kv head
  pdl_wait();
  pdl_trigger();

  int k0 = kp * KC;
  float rr[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) rr[j] = __ldg(a.R_K + (k0 + j) * D + col);
  for (int idx = threadIdx.x; idx < G * D; idx += kQrotThreads)
    qs[idx / D][idx % D] = a.in_fp32 ? static_cast<const float*>(a.q)[q0 + idx]
                                     : __bfloat162float(static_cast<const __nv_bfloat16*>(a.q)[q0 + idx]);
  __syncthreads();
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
  for (;;) {
#pragma unroll
    for (int j = 0; j < 32; ++j)
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (i < G) acc[i] = fmaf(qs[i][k0 + j], rr[j], acc[i]);
    k0 += 32;
    if (k0 >= (kp + 1) * KC) break;
#pragma unroll
    for (int j = 0; j < 32; ++j) rr[j] = __ldg(a.R_K + (k0 + j) * D + col);
  }
  if (kp > 0) {
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (i < G) part[kp - 1][i][c] = acc[i];
  }
  if (chunk == 0 && threadIdx.x == 0) a.ticket[bh] = 0;
  __syncthreads();
  if (kp == 0) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (i < G) {
        float sum = acc[i];
#pragma unroll
        for (int p = 0; p < KP - 1; ++p) sum += part[p][i][c];
        const float v = sum * a.qscale;
        if (!(fabsf(v) < 60000.f)) status_or(a.status, OSCAR_DEV_FP16_RANGE);
        a.qprime[q0 + i * D + col] = v;
        float t = v;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
        if ((c & 31) == 0) red[i][c >> 5] = t;
      }
    }
  }
  __syncthreads();
  if (threadIdx.x < G)
    a.qsum[(q0 / D + threadIdx.x) * (D / kGroup) + chunk] =
        red[threadIdx.x][0] + red[threadIdx.x][1] + red[threadIdx.x][2] + red[threadIdx.x][3];
}

// ---------------------------------------------------------------------------
// split kernel
// ---------------------------------------------------------------------------
template <int D, int NQT>
__global__ void __launch_bounds__(kThreads, (D == 128 ? 2 : 1))
    split_kernel(const __grid_constant__ CUtensorMap tks, const __grid_constant__ CUtensorMap tvs,
                 const __grid_constant__ CUtensorMap tkr, const __grid_constant__ CUtensorMap tvr,
                 const DecodeArgs a) {
  using C = DecCfg<D, NQT>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 128-byte-swizzled TMA destinations need 1 KB alignment
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  __shared__ int abort_flag;

  const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const Geom& g = a.g;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int T = clamp_seq_len(a, b);
  const Regions rg = make_regions(T, g.S, g.W, D);
  const int64_t total = rg.nsb * rg.cbf + rg.nib * rg.ci2 + rg.nrb * rg.cbf;
  const int kb = first_block_at(rg, (int64_t(split) * total + a.ns - 1) / a.ns);
  const int ke = first_block_at(rg, (int64_t(split + 1) * total + a.ns - 1) / a.ns);
  const int nblk = ke - kb;
  const int64_t bh = int64_t(b) * g.Hkv + h;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int s = 0; s < C::NST; ++s) mbar_init(smem_u32(&bars[s]), 1);  // issuer's arrival + tx bytes
    mbar_init(smem_u32(&bars[C::NST]), 1);  // R_V prefetch of the merging CTA
    mbar_fence_init();
  }
  __syncthreads();

  const uint8_t* kbase = a.layer_base;
  const uint8_t* vbase = a.layer_base + g.role_bytes;
  const uint64_t codes_off = g.sink_bytes + g.ring_bytes;
  const uint64_t sz_off = codes_off + g.codes_bytes;

  // Bulk copies of block kl into stage `stage`, issued by the calling warp (lane
  // 0 arms the barrier with the byte count first).
  auto issue_block = [&](int kl, int stage) {
    const Blk bk = block_at(rg, kb + kl);
    const uint32_t full = smem_u32(&bars[stage]);
    const uint32_t dst = smem_u32(smem + C::OFF_STAGE + stage * C::STAGE);
    if (bk.type == 1) {
      if (lane == 0) {
        const int n4 = (bk.count + 3) & ~3;
        const uint32_t cb = n4 * C::ROWB, sb = n4 * C::Dg * 4;
        mbar_arrive_expect_tx(full, 2 * cb + 2 * sb);
        const int64_t row = bh * g.ncap + bk.first;
        bulk_g2s(dst, kbase + codes_off + row * C::ROWB, cb, full);
        bulk_g2s(dst + kI2Tok * C::ROWB, vbase + codes_off + row * C::ROWB, cb, full);
        bulk_g2s(dst + 2 * kI2Tok * C::ROWB, kbase + sz_off + row * C::Dg * 4, sb, full);
        bulk_g2s(dst + 2 * kI2Tok * C::ROWB + kI2Tok * C::Dg * 4, vbase + sz_off + row * C::Dg * 4, sb, full);
      }
    } else {
      // 16 rows of K and V as 64-column boxes, 128-byte swizzled by the TMA unit
      if (lane == 0) {
        mbar_arrive_expect_tx(full, 2 * C::BOXES * C::BOX_BYTES);
        const CUtensorMap* mk = bk.type == 0 ? &tks : &tkr;
        const CUtensorMap* mv = bk.type == 0 ? &tvs : &tvr;
        const int row0 = int(bk.type == 0 ? bh * g.S + bk.first : bh * g.W + bk.first);
#pragma unroll
        for (int q = 0; q < C::BOXES; ++q) {
          tma_load_2d(dst + q * C::BOX_BYTES, mk, 64 * q, row0, full);
          tma_load_2d(dst + (C::BOXES + q) * C::BOX_BYTES, mv, 64 * q, row0, full);
        }
      }
    }
  };

  // ------------------------------- consumers --------------------------------
  const int team = warp / C::TS, wt = warp % C::TS;  // wt = quant group handled
  const int gq = lane >> 2, cq = lane & 3;
  const int Gh = g.G;
  const int head0 = h * Gh;  // first query head of this kv head
  const int nmine = nblk > team ? (nblk - team + C::NTEAMS - 1) / C::NTEAMS : 0;  // this team's blocks
  auto my_stage = [&](int j) { return team * C::NSTW + j % C::NSTW; };
  int issued = 0;  // blocks of this team whose copies are in flight or done

  // the cache is complete once this kernel runs (the preceding kernel waited
  // for it); start streaming before waiting for q'
  if (wt == 0)
    for (; issued < nmine && issued < C::NSTW; ++issued) issue_block(team + issued * C::NTEAMS, my_stage(issued));

  pdl_wait();  // q' comes from the preceding kernel

  // B fragments of q' for this warp's group: column n <-> (head n/2, hi|lo by n%2).
  // INT2 codes reach the MMAs as fp16 subnormals code * 4^k * 2^-24 (see
  // unpack16), so the q' entry meeting a code at mantissa bit 2k is stored as
  // q' * 4^-k * 2^X, with 2^X per (head, group) chosen so that the largest
  // |q'| * 2^X lies in [2^13, 2^14): every product is then code * q' * 2^(X-24)
  // and the score is rescaled by qF = 2^(24-X) (exact powers of two throughout).
  uint32_t qf[8][NQT][2];
  float qsum[NQT], qF[NQT];
  // bf16 B fragments for BF16 blocks: n-tile 2nq holds (hi, mid) and n-tile
  // 2nq+1 holds (lo, 0) of each head's three-way bf16 split (~24 bits)
  uint32_t* qbf = reinterpret_cast<uint32_t*>(smem + C::OFF_QBF) + wt * 8 * C::NQB * 64;
  {
    const int hs_b = gq >> 1, lohalf = gq & 1;
#pragma unroll
    for (int nq = 0; nq < NQT; ++nq) {
      const int hb = 4 * nq + hs_b;  // head slot of this lane's B column
      const bool hv = hb < Gh;
      const float* qp = a.qprime + (int64_t(b) * g.Hq + head0 + (hv ? hb : 0)) * D + wt * kGroup;
      float xq[8][2][2];
      float mx = 0.f;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const int d0 = 16 * kk + 2 * cq + 8 * half;
          xq[kk][half][0] = hv ? qp[d0] : 0.f;
          xq[kk][half][1] = hv ? qp[d0 + 1] : 0.f;
          mx = fmaxf(mx, fmaxf(fabsf(xq[kk][half][0]), fabsf(xq[kk][half][1])));
        }
      // the four lanes of a B column hold all 128 channels of the group
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      int ex = 0;
      (void)frexpf(mx, &ex);  // mx < 2^ex
      const int X = mx > 0.f ? min(14 - ex, 100) : 0;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const float f = ldexpf(1.f, X - 2 * unpack_k(2 * (kk & 3) + half));
          const float x0 = xq[kk][half][0], x1 = xq[kk][half][1];
          const uint32_t s0 = split_f16(x0 * f), s1 = split_f16(x1 * f);
          // pick hi (low half) or lo (high half) of each split
          const uint32_t v16 = lohalf ? ((s0 >> 16) | (s1 & 0xffff0000u)) : ((s0 & 0xffffu) | (s1 << 16));
          qf[kk][nq][half] = v16;
          if (team == 0) {  // the other teams hold the same fragments
            uint32_t p0[3], p1[3];
            split3_bf16(x0, p0);
            split3_bf16(x1, p1);
            const uint32_t va = lohalf ? (p0[1] | (p1[1] << 16)) : (p0[0] | (p1[0] << 16));
            const uint32_t vb = lohalf ? 0u : (p0[2] | (p1[2] << 16));
            qbf[(kk * C::NQB + 2 * nq) * 64 + half * 32 + lane] = va;
            qbf[(kk * C::NQB + 2 * nq + 1) * 64 + half * 32 + lane] = vb;
          }
        }
      }
      const int hc = 4 * nq + cq;  // head owned by this lane in C fragments
      // lane 8 * cq holds B column 2 * cq, i.e. head slot cq of this n-tile
      qF[nq] = ldexpf(1.f, 24 - __shfl_sync(0xffffffffu, X, 8 * cq));
      qsum[nq] = hc < Gh ? a.qsum[(int64_t(b) * g.Hq + head0 + hc) * C::Dg + wt] : 0.f;
    }
  }
  __syncwarp();

  asm volatile("bar.sync 14, %0;" ::"r"(32 * kNCW) : "memory");  // shared bf16 fragments written

  float o[8][NQT][4];
  float m_run[NQT], l_run[NQT], zeta[NQT];
#pragma unroll
  for (int nq = 0; nq < NQT; ++nq) {
    m_run[nq] = -INFINITY; l_run[nq] = 0.f; zeta[nq] = 0.f;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
      for (int e = 0; e < 4; ++e) o[mt][nq][e] = 0.f;
  }

  float* xch = reinterpret_cast<float*>(smem + C::OFF_XCH);
  int xbuf = 0;

  // INT2 P.V takes V codes from unpack16_v: the code of output row r arrives
  // as code * 2^e(r), e(r) = unpack_v_exp(p) with p = 2 * (mtd % 4) for rows gq
  // and 2 * (mtd % 4) + 1 for rows gq + 8.  While INT2 blocks are consumed, row
  // r of o holds (real value) * 2^e(r); it is converted by exact powers of two
  // at a switch between INT2 and BF16 blocks and at the end.
  bool o_i2 = false;
  auto scale_o = [&](int sign) {  // o *= 2^(sign * e(r)) per row
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      const float f0 = ldexpf(1.f, sign * unpack_v_exp(2 * (mt & 3)));
      const float f1 = ldexpf(1.f, sign * unpack_v_exp(2 * (mt & 3) + 1));
#pragma unroll
      for (int nq = 0; nq < NQT; ++nq) {
        o[mt][nq][0] *= f0; o[mt][nq][1] *= f0;
        o[mt][nq][2] *= f1; o[mt][nq][3] *= f1;
      }
    }
  };


  for (int j = 0; j < nmine; ++j) {
    const int kl = team + j * C::NTEAMS;
    const int stage = my_stage(j);
    int ok = 1;
    if (lane == 0) ok = mbar_wait(smem_u32(&bars[stage]), (j / C::NSTW) & 1);
    ok = __shfl_sync(0xffffffffu, ok, 0);
    // the warps of a team must take the same decision: they meet at team barriers below
    if constexpr (C::TS > 1) ok = team_all(ok, 1 + team, 32 * C::TS);
    if (!ok) {
      if (lane == 0) { abort_flag = 1; status_or(a.status, OSCAR_DEV_TIMEOUT); }
      break;
    }
    const Blk bk = block_at(rg, kb + kl);
    const uint8_t* st = smem + C::OFF_STAGE + stage * C::STAGE;
    const bool is_i2 = bk.type == 1;
    if (is_i2 != o_i2) {
      scale_o(is_i2 ? 1 : -1);
      o_i2 = is_i2;
    }
    constexpr int MT_MAX = kSub / 16;
    const int nmt = is_i2 ? MT_MAX : 1;
    const int nsub = is_i2 ? (bk.count + kSub - 1) / kSub : 1;
    for (int sbk = 0; sbk < nsub; ++sbk) {
    const int cnt = is_i2 ? min(kSub, bk.count - sbk * kSub) : bk.count;  // tokens in this sub-block
    const int tb = sbk * kSub;  // its first token within the stage

    // ---- scores: s[mt][nq][0] token 16mt+gq, [1] token 16mt+gq+8
    float s[MT_MAX][NQT][2];
    float ksc[MT_MAX][2], kze[MT_MAX][2];
    if (is_i2) {
      const uint8_t* kc = st;
      const uint32_t* ksz = reinterpret_cast<const uint32_t*>(st + 2 * kI2Tok * C::ROWB);
      // m-tiles are processed in groups whose MMAs interleave (independent
      // accumulators), so the k-step chain of one m-tile never runs alone
      constexpr int MG = NQT == 1 ? 4 : 2;
#pragma unroll
      for (int m0 = 0; m0 < MT_MAX; m0 += MG) {
        uint2 w[MG][2];
#pragma unroll
        for (int i = 0; i < MG; ++i) {
          const int t0 = 16 * (m0 + i) + gq;
          w[i][0] = *reinterpret_cast<const uint2*>(kc + (tb + t0) * C::ROWB + wt * 32 + cq * 8);
          w[i][1] = *reinterpret_cast<const uint2*>(kc + (tb + t0 + 8) * C::ROWB + wt * 32 + cq * 8);
        }
        float acc[MG][NQT][4];
#pragma unroll
        for (int i = 0; i < MG; ++i)
#pragma unroll
          for (int nq = 0; nq < NQT; ++nq)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[i][nq][e] = 0.f;
#pragma unroll
        for (int wi = 0; wi < 2; ++wi) {
          uint32_t r[MG][2][8];
#pragma unroll
          for (int i = 0; i < MG; ++i) {
            unpack16(wi ? w[i][0].y : w[i][0].x, r[i][0]);
            unpack16(wi ? w[i][1].y : w[i][1].x, r[i][1]);
          }
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4) {
            const int kk = 4 * wi + k4;
#pragma unroll
            for (int nq = 0; nq < NQT; ++nq)
#pragma unroll
              for (int i = 0; i < MG; ++i)
                mma_f16(acc[i][nq], r[i][0][2 * k4], r[i][1][2 * k4], r[i][0][2 * k4 + 1], r[i][1][2 * k4 + 1],
                        qf[kk][nq][0], qf[kk][nq][1]);
          }
        }
#pragma unroll
        for (int i = 0; i < MG; ++i) {
          const int mt = m0 + i;
          const int t0 = 16 * mt + gq, t1 = t0 + 8;
          const uint32_t z0 = ksz[(tb + t0) * C::Dg + wt], z1 = ksz[(tb + t1) * C::Dg + wt];
          ksc[mt][0] = __half2float(__ushort_as_half(z0 & 0xffff));
          kze[mt][0] = __half2float(__ushort_as_half(z0 >> 16));
          ksc[mt][1] = __half2float(__ushort_as_half(z1 & 0xffff));
          kze[mt][1] = __half2float(__ushort_as_half(z1 >> 16));
#pragma unroll
          for (int nq = 0; nq < NQT; ++nq) {
            s[mt][nq][0] = fmaf(ksc[mt][0], (acc[i][nq][0] + acc[i][nq][1]) * qF[nq], kze[mt][0] * qsum[nq]);
            s[mt][nq][1] = fmaf(ksc[mt][1], (acc[i][nq][2] + acc[i][nq][3]) * qF[nq], kze[mt][1] * qsum[nq]);
          }
        }
      }
    } else {
      const uint32_t kb_s = smem_u32(st);
      float acc[C::NQB][4];
#pragma unroll
      for (int nb = 0; nb < C::NQB; ++nb)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[nb][e] = 0.f;
      const int mi = lane >> 3;
      const int tok = (lane & 7) + 8 * (mi & 1);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const int dim = wt * kGroup + 16 * kk + 8 * (mi >> 1);
        uint32_t a0, a1, a2, a3;
        ldmatrix_x4(kb_s + (dim >> 6) * C::BOX_BYTES + tok * 128 + ((((dim & 63) >> 3) ^ (tok & 7)) << 4), a0, a1,
                    a2, a3);
#pragma unroll
        for (int nb = 0; nb < C::NQB; ++nb) {
          const uint32_t b0 = qbf[(kk * C::NQB + nb) * 64 + lane];
          const uint32_t b1 = qbf[(kk * C::NQB + nb) * 64 + 32 + lane];
          mma_bf16(acc[nb], a0, a1, a2, a3, b0, b1);
        }
      }
#pragma unroll
      for (int nq = 0; nq < NQT; ++nq) {
        s[0][nq][0] = acc[2 * nq][0] + acc[2 * nq][1] + acc[2 * nq + 1][0];
        s[0][nq][1] = acc[2 * nq][2] + acc[2 * nq][3] + acc[2 * nq + 1][2];
      }
    }

    // ---- team exchange of partial scores (one quant group per warp)
    if constexpr (C::TS > 1) {
      float* xb = xch + ((team * 2 + xbuf) * C::TS) * kSub * C::HEADS;
#pragma unroll
      for (int mt = 0; mt < MT_MAX; ++mt) {
        if (mt < nmt) {
#pragma unroll
          for (int nq = 0; nq < NQT; ++nq) {
            const int hs = 4 * nq + cq;
            xb[(wt * kSub + 16 * mt + gq) * C::HEADS + hs] = s[mt][nq][0];
            xb[(wt * kSub + 16 * mt + gq + 8) * C::HEADS + hs] = s[mt][nq][1];
          }
        }
      }
      asm volatile("bar.sync %0, %1;" ::"r"(1 + team), "r"(32 * C::TS) : "memory");
#pragma unroll
      for (int mt = 0; mt < MT_MAX; ++mt) {
        if (mt < nmt) {
#pragma unroll
          for (int nq = 0; nq < NQT; ++nq) {
            const int hs = 4 * nq + cq;
            float t0 = 0.f, t1 = 0.f;
#pragma unroll
            for (int w = 0; w < C::TS; ++w) {
              t0 += xb[(w * kSub + 16 * mt + gq) * C::HEADS + hs];
              t1 += xb[(w * kSub + 16 * mt + gq + 8) * C::HEADS + hs];
            }
            s[mt][nq][0] = t0;
            s[mt][nq][1] = t1;
          }
        }
      }
      xbuf ^= 1;
    }

    // ---- online softmax (log2 units)
    float p[MT_MAX][NQT][2];
#pragma unroll
    for (int nq = 0; nq < NQT; ++nq) {
      float mb = -INFINITY;
#pragma unroll
      for (int mt = 0; mt < MT_MAX; ++mt) {
        if (mt < nmt) {
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int tk = 16 * mt + gq + 8 * e;
            const float v = tk < cnt ? s[mt][nq][e] : -INFINITY;
            s[mt][nq][e] = v;
            mb = fmaxf(mb, v);
          }
        }
      }
      mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 4));
      mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 8));
      mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 16));
      const float mnew = fmaxf(m_run[nq], mb);
      const float corr = ex2(m_run[nq] - mnew);  // 0 on the first block
      m_run[nq] = mnew;
      if (__any_sync(0xffffffffu, corr != 1.f)) {
        l_run[nq] *= corr;
        zeta[nq] *= corr;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt)
#pragma unroll
          for (int e = 0; e < 4; ++e) o[mt][nq][e] *= corr;
      }
#pragma unroll
      for (int mt = 0; mt < MT_MAX; ++mt) {
        if (mt < nmt) {
          p[mt][nq][0] = ex2(s[mt][nq][0] - mnew);
          p[mt][nq][1] = ex2(s[mt][nq][1] - mnew);
          l_run[nq] += p[mt][nq][0] + p[mt][nq][1];
        }
      }
    }

    // ---- P.V
    if (is_i2) {
      const uint32_t* vc = reinterpret_cast<const uint32_t*>(st + kI2Tok * C::ROWB);
#pragma unroll
      for (int ks = 0; ks < MT_MAX; ++ks) {
        uint32_t bw0[NQT], bw1[NQT];
        // V scale/zero of this lane's two tokens (group wt)
        const uint32_t* vsz = reinterpret_cast<const uint32_t*>(st + 2 * kI2Tok * C::ROWB) + kI2Tok * C::Dg;
        const int t0 = 16 * ks + gq, t1 = t0 + 8;
        const uint32_t z0 = vsz[(tb + t0) * C::Dg + wt], z1 = vsz[(tb + t1) * C::Dg + wt];
        const float vs0 = __half2float(__ushort_as_half(z0 & 0xffff));
        const float vz0 = __half2float(__ushort_as_half(z0 >> 16));
        const float vs1 = __half2float(__ushort_as_half(z1 & 0xffff));
        const float vz1 = __half2float(__ushort_as_half(z1 >> 16));
        const bool v0 = t0 < cnt, v1 = t1 < cnt;
#pragma unroll
        for (int nq = 0; nq < NQT; ++nq) {
          const float w0 = v0 ? p[ks][nq][0] * vs0 : 0.f;
          const float w1 = v1 ? p[ks][nq][1] * vs1 : 0.f;
          zeta[nq] += (v0 ? p[ks][nq][0] * vz0 : 0.f) + (v1 ? p[ks][nq][1] * vz1 : 0.f);
          bw0[nq] = movmatrix_trans(split_f16(w0));
          bw1[nq] = movmatrix_trans(split_f16(w1));
        }
        // codes of word (wt, gq) for tokens 2cq, 2cq+1, 2cq+8, 2cq+9 of this k-step
        const int ta = 16 * ks + 2 * cq;
        const uint32_t wa = vc[(tb + ta + 0) * (C::ROWB / 4) + wt * 8 + gq];
        const uint32_t wb = vc[(tb + ta + 1) * (C::ROWB / 4) + wt * 8 + gq];
        const uint32_t wc = vc[(tb + ta + 8) * (C::ROWB / 4) + wt * 8 + gq];
        const uint32_t wd = vc[(tb + ta + 9) * (C::ROWB / 4) + wt * 8 + gq];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          uint32_t rx[8], ry[8];
          unpack16_v(prmt(wa, wb, hh ? 0x7632u : 0x5410u), rx);
          unpack16_v(prmt(wc, wd, hh ? 0x7632u : 0x5410u), ry);
#pragma unroll
          for (int m4 = 0; m4 < 4; ++m4) {
            const int mtd = 4 * hh + m4;
#pragma unroll
            for (int nq = 0; nq < NQT; ++nq)
              mma_f16(o[mtd][nq], rx[2 * m4], rx[2 * m4 + 1], ry[2 * m4], ry[2 * m4 + 1], bw0[nq], bw1[nq]);
          }
        }
      }
    } else {
      uint32_t bw0[NQT], bw1[NQT];
#pragma unroll
      for (int nq = 0; nq < NQT; ++nq) {
        bw0[nq] = movmatrix_trans(split_bf16(p[0][nq][0]));
        bw1[nq] = movmatrix_trans(split_bf16(p[0][nq][1]));
      }
      const uint32_t vb_s = smem_u32(st + C::BOXES * C::BOX_BYTES);
      const int mi = lane >> 3;
      const int tok = (lane & 7) + 8 * (mi >> 1);
      const bool partial = cnt < kBfTok;
      // tokens held by this lane's A fragment halves
      const bool va = 2 * cq < cnt, vb = 2 * cq + 1 < cnt;
      const bool vc8 = 2 * cq + 8 < cnt, vd = 2 * cq + 9 < cnt;
      const uint32_t mask01 = (va ? 0xffffu : 0u) | (vb ? 0xffff0000u : 0u);
      const uint32_t mask89 = (vc8 ? 0xffffu : 0u) | (vd ? 0xffff0000u : 0u);
#pragma unroll
      for (int mtd = 0; mtd < 8; ++mtd) {
        const int dim = wt * kGroup + 16 * mtd + 8 * (mi & 1);
        uint32_t a0, a1, a2, a3;
        ldmatrix_x4_trans(vb_s + (dim >> 6) * C::BOX_BYTES + tok * 128 + ((((dim & 63) >> 3) ^ (tok & 7)) << 4),
                          a0, a1, a2, a3);
        if (partial) {
          a0 &= mask01; a1 &= mask01; a2 &= mask89; a3 &= mask89;
        }
#pragma unroll
        for (int nq = 0; nq < NQT; ++nq) mma_bf16(o[mtd][nq], a0, a1, a2, a3, bw0[nq], bw1[nq]);
      }
    }
    }  // sub-blocks

    // every warp of the team is done with this stage: refill it
    if constexpr (C::TS > 1) {
      asm volatile("bar.sync %0, %1;" ::"r"(1 + team), "r"(32 * C::TS) : "memory");
    } else {
      __syncwarp();
    }
    if (wt == 0 && issued < nmine) {
      issue_block(team + issued * C::NTEAMS, my_stage(issued));
      ++issued;
    }
  }
  if (o_i2) scale_o(-1);
  // after an early exit, wait (bounded) for copies still landing in our stages
  if (wt == 0 && lane == 0) {
    const int consumed = *((volatile int*)&abort_flag) ? 0 : nmine;
    for (int jj = (issued > C::NSTW ? issued - C::NSTW : 0); jj < issued; ++jj)
      if (jj >= consumed && !mbar_wait(smem_u32(&bars[my_stage(jj)]), (jj / C::NSTW) & 1)) break;
  }

  // ---- team partials -> shared memory
#pragma unroll
  for (int nq = 0; nq < NQT; ++nq) {
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      l_run[nq] += __shfl_xor_sync(0xffffffffu, l_run[nq], off);
      zeta[nq] += __shfl_xor_sync(0xffffffffu, zeta[nq], off);
    }
  }
  float* part = reinterpret_cast<float*>(smem + C::OFF_PART);  // [team][head][D + 2]
#pragma unroll
  for (int nq = 0; nq < NQT; ++nq) {
    const int hs = 4 * nq + cq;
    float* ph = part + (team * C::HEADS + hs) * (D + 2);
#pragma unroll
    for (int mtd = 0; mtd < 8; ++mtd) {
      const int d0 = wt * kGroup + 16 * mtd + gq;
      ph[d0] = o[mtd][nq][0] + o[mtd][nq][1] + zeta[nq];
      ph[d0 + 8] = o[mtd][nq][2] + o[mtd][nq][3] + zeta[nq];
    }
    if (wt == 0 && gq == 0) {
      ph[D] = m_run[nq];
      ph[D + 1] = l_run[nq];
    }
  }
  asm volatile("bar.sync 15, %0;" ::"r"(32 * kNCW) : "memory");
  pdl_trigger();

  // ---- merge the teams of this CTA and write the split partial
  for (int idx = threadIdx.x; idx < Gh * D; idx += 32 * kNCW) {
    const int hs = idx / D, d = idx % D;
    float M = -INFINITY;
#pragma unroll
    for (int t = 0; t < C::NTEAMS; ++t) M = fmaxf(M, part[(t * C::HEADS + hs) * (D + 2) + D]);
    float acc = 0.f, L = 0.f;
#pragma unroll
    for (int t = 0; t < C::NTEAMS; ++t) {
      const float* ph = part + (t * C::HEADS + hs) * (D + 2);
      const float w = M == -INFINITY ? 0.f : ex2(ph[D] - M);
      acc += w * ph[d];
      L += w * ph[D + 1];
    }
    const int64_t pi = (int64_t(b) * g.Hq + head0 + hs) * a.ns + split;
    a.ws_acc[pi * D + d] = acc;
    if (d == 0) {
      a.ws_ml[pi * 2 + 0] = M;
      a.ws_ml[pi * 2 + 1] = L;
    }
  }

  // ---- the last CTA of this (b, kv head) to finish merges all splits (a ticket,
  // no waiting on other CTAs), un-rotates V and stores the output
  __shared__ int is_last;
  __threadfence();
  asm volatile("bar.sync 15, %0;" ::"r"(32 * kNCW) : "memory");
  if (threadIdx.x == 0) is_last = atomicAdd(a.ticket + bh, 1) == a.ns - 1;
  asm volatile("bar.sync 15, %0;" ::"r"(32 * kNCW) : "memory");
  if (!is_last) return;
  __threadfence();
  // D = 128: prefetch R_V (64 KB) into the now idle stage area with one bulk copy
  constexpr bool kRvSmem = D == 128 && !(C::NST * C::STAGE < D * D * 4);
  const float* rvs = reinterpret_cast<const float*>(smem + C::OFF_STAGE);
  const uint32_t rv_bar = smem_u32(&bars[C::NST]);
  if constexpr (kRvSmem) {
    if (threadIdx.x == 0 && !a.absorb_v) {
      mbar_arrive_expect_tx(rv_bar, D * D * 4);
      bulk_g2s(smem_u32(smem + C::OFF_STAGE), a.R_V, D * D * 4, rv_bar);
    }
  }
  float* ob = part;                    // [G][D] merged o' (rotated basis)
  float* Ms = part + C::HEADS * D;     // [G] max, [G] sum
  float* Ls = Ms + C::HEADS;
  float* wts = Ls + C::HEADS;          // [G][splits] normalised split weights
  for (int i = warp; i < Gh; i += kNCW) {
    const int64_t base = (int64_t(b) * g.Hq + head0 + i) * a.ns;
    const float m0 = lane < a.ns ? __ldcg(a.ws_ml + (base + lane) * 2) : -INFINITY;
    const float l0 = lane < a.ns ? __ldcg(a.ws_ml + (base + lane) * 2 + 1) : 0.f;
    const float m1 = lane + 32 < a.ns ? __ldcg(a.ws_ml + (base + lane + 32) * 2) : -INFINITY;
    const float l1 = lane + 32 < a.ns ? __ldcg(a.ws_ml + (base + lane + 32) * 2 + 1) : 0.f;
    float M = fmaxf(m0, m1);
#pragma unroll
    for (int o2 = 16; o2 > 0; o2 >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o2));
    const float e0 = M == -INFINITY || m0 == -INFINITY ? 0.f : ex2(m0 - M);
    const float e1 = M == -INFINITY || m1 == -INFINITY ? 0.f : ex2(m1 - M);
    float L = e0 * l0 + e1 * l1;
#pragma unroll
    for (int o2 = 16; o2 > 0; o2 >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o2);
    const float inv = L > 0.f ? 1.f / L : 0.f;
    if (lane < a.ns) wts[i * OSCAR_KV_MAX_SPLITS + lane] = e0 * inv;
    if (lane + 32 < a.ns) wts[i * OSCAR_KV_MAX_SPLITS + lane + 32] = e1 * inv;
    if (lane == 0) {
      Ms[i] = M;
      Ls[i] = L;
    }
  }
  asm volatile("bar.sync 15, %0;" ::"r"(32 * kNCW) : "memory");
  for (int idx = threadIdx.x; idx < Gh * D; idx += 32 * kNCW) {
    const int i = idx / D, d = idx % D;
    const int64_t base = (int64_t(b) * g.Hq + head0 + i) * a.ns;
    const float* wi = wts + i * OSCAR_KV_MAX_SPLITS;
    float acc = 0.f;
#pragma unroll 8
    for (int sp = 0; sp < a.ns; ++sp) acc = fmaf(wi[sp], __ldcg(a.ws_acc + (base + sp) * D + d), acc);
    ob[idx] = acc;
  }
  asm volatile("bar.sync 15, %0;" ::"r"(32 * kNCW) : "memory");
  bool rv_ok = true;
  if constexpr (kRvSmem) {
    if (!a.absorb_v) rv_ok = mbar_wait(rv_bar, 0);
    if (!rv_ok && threadIdx.x == 0) status_or(a.status, OSCAR_DEV_TIMEOUT);
  }
  // o = o' R_V^T: o[r] = sum_j R_V[r][j] o'[j]; one thread per output channel r
  for (int r = threadIdx.x; r < D; r += 32 * kNCW) {
    float res[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) res[i] = 0.f;
    if (a.absorb_v) {
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (i < Gh) res[i] = ob[i * D + r];
    } else if (kRvSmem && rv_ok) {
      // skewed walk over j: thread r touches bank (r + jj) % 32, no conflicts
#pragma unroll 4
      for (int jj = 0; jj < D; ++jj) {
        const int j = (jj + r) & (D - 1);
        const float rv = rvs[r * D + j];
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if (i < Gh) res[i] = fmaf(rv, ob[i * D + j], res[i]);
      }
    } else {
      const float4* rv4 = reinterpret_cast<const float4*>(a.R_V + int64_t(r) * D);
#pragma unroll 8
      for (int j4 = 0; j4 < D / 4; ++j4) {
        const float4 rv = __ldg(rv4 + j4);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if (i < Gh) {
            const float* oi = ob + i * D + 4 * j4;
            res[i] = fmaf(rv.x, oi[0], fmaf(rv.y, oi[1], fmaf(rv.z, oi[2], fmaf(rv.w, oi[3], res[i]))));
          }
        }
      }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (i < Gh) {
        const int64_t oi = (int64_t(b) * g.Hq + head0 + i) * D + r;
        if (a.out_fp32)
          static_cast<float*>(a.out)[oi] = res[i];
        else
          static_cast<__nv_bfloat16*>(a.out)[oi] = __float2bfloat16_rn(res[i]);
      }
    }
  }
  if (threadIdx.x < Gh) {
    const int i = threadIdx.x;
    if (a.lse) {
      const float M = Ms[i], L = Ls[i];
      a.lse[int64_t(b) * g.Hq + head0 + i] =
          (M == -INFINITY || !(L > 0.f)) ? -INFINITY : (M + log2f(L)) * 0.6931471805599453f;
    }
    if (i == 0 && h == 0) {
      if (a.seq_lens[b] > g.cap) status_or(a.status, OSCAR_DEV_OVER_CAPACITY);
      if (T < 1) status_or(a.status, OSCAR_DEV_EMPTY);
    }
  }
}

// ---------------------------------------------------------------------------
// host launch
// ---------------------------------------------------------------------------
template <typename K, typename... Args>
cudaError_t launch_pdl(K kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t stream, const Args&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

struct DevInfo {
  int sms = 0;
  int occ[3][2] = {{0, 0}, {0, 0}, {0, 0}};
  bool ready = false;
};
DevInfo g_dev[64];

template <int D, int NQT>
int prepare_split(int dev) {
  using C = DecCfg<D, NQT>;
  if (cudaFuncSetAttribute(split_kernel<D, NQT>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) !=
      cudaSuccess)
    return -1;
  int occ = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, split_kernel<D, NQT>, kThreads, C::SMEM) !=
      cudaSuccess)
    return -1;
  return occ;
}

int dinfo_init(int dev) {
  DevInfo& di = g_dev[dev];
  if (di.ready) return 0;
  if (cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
  const int o[6] = {prepare_split<128, 1>(dev), prepare_split<128, 2>(dev), prepare_split<256, 1>(dev),
                    prepare_split<256, 2>(dev), prepare_split<512, 1>(dev), prepare_split<512, 2>(dev)};
  for (int i = 0; i < 6; ++i) {
    if (o[i] <= 0) return -1;
    di.occ[i / 2][i % 2] = o[i];
  }
  di.ready = true;
  return 0;
}

int didx(int D) { return D == 128 ? 0 : (D == 256 ? 1 : 2); }

template <int D, int NQT>
int launch_decode_d(const DecodeArgs& a, cudaStream_t stream) {
  using C = DecCfg<D, NQT>;
  const Geom& g = a.g;
  if (launch_pdl(qrot_kernel<D>, dim3(g.B * g.Hkv, D / 128), dim3(kQrotThreads), 0, stream, a) != cudaSuccess) return OSCAR_ERR_LAUNCH;
  const bool prof = g_prof_start != nullptr && g_prof_stop != nullptr;
  if (prof && cudaEventRecord(g_prof_start, stream) != cudaSuccess) return OSCAR_ERR_LAUNCH;
  // TMA maps of this layer's BF16 windows: [B*Hkv*S][D] sink and [B*Hkv*W][D] ring, per role
  CUtensorMap maps[4];
  std::memset(maps, 0, sizeof(maps));
  const uint8_t* kb = a.layer_base;
  const uint8_t* vb = a.layer_base + g.role_bytes;
  const uint64_t bh = uint64_t(g.B) * g.Hkv;
  if (g.S > 0 && (!encode_rows_bf16(&maps[0], kb, bh * g.S, D, 64, kBfTok) ||
                  !encode_rows_bf16(&maps[1], vb, bh * g.S, D, 64, kBfTok)))
    return OSCAR_ERR_LAUNCH;
  if (g.W > 0 && (!encode_rows_bf16(&maps[2], kb + g.sink_bytes, bh * g.W, D, 64, kBfTok) ||
                  !encode_rows_bf16(&maps[3], vb + g.sink_bytes, bh * g.W, D, 64, kBfTok)))
    return OSCAR_ERR_LAUNCH;
  if (launch_pdl(split_kernel<D, NQT>, dim3(a.ns, g.Hkv, g.B), dim3(kThreads), C::SMEM, stream, maps[0], maps[1],
                 maps[2], maps[3], a) != cudaSuccess)
    return OSCAR_ERR_LAUNCH;
  if (prof && cudaEventRecord(g_prof_stop, stream) != cudaSuccess) return OSCAR_ERR_LAUNCH;
  return OSCAR_OK;
}

}  // namespace

thread_local cudaEvent_t g_prof_start = nullptr, g_prof_stop = nullptr;

uint64_t decode_workspace_bytes(const Geom& g, int ns) {
  const uint64_t bq = uint64_t(g.B) * g.Hq;
  return align256(bq * g.D * 4) + align256(bq * g.Dg * 4) + align256(bq * ns * g.D * 4) +
         align256(bq * ns * 2 * 4) + align256(uint64_t(g.B) * g.Hkv * 4);
}

int decode_auto_splits(const Geom& g, int seq_len_hint) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev >= 64 || dinfo_init(dev) != 0) return -1;
  const DevInfo& di = g_dev[dev];
  const int occ = di.occ[didx(g.D)][g.G > 4 ? 1 : 0];
  const int slots = di.sms * occ;
  const int units = g.B * g.Hkv;
  // at least ~2 INT2 blocks of work per split
  const int max_by_len = std::max(1, seq_len_hint / (2 * kI2Tok));
  // best wave efficiency with at most two waves; a second wave must pay for its
  // extra start-up and merge work with a clearly better fill
  int best = 1;
  double best_eff = -1.0;
  const int cap = std::min(max_by_len, int(OSCAR_KV_MAX_SPLITS));
  for (int ns = 1; ns <= cap; ++ns) {
    const int64_t ctas = int64_t(ns) * units;
    const int64_t waves = (ctas + slots - 1) / slots;
    if (waves > 2) break;
    const double eff = double(ctas) / double(waves * slots) - (waves > 1 ? 0.05 : 0.0);
    if (eff > best_eff + 1e-9) {
      best_eff = eff;
      best = ns;
    }
  }
  return best;
}

int launch_decode(const DecodeArgs& a, cudaStream_t stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev >= 64 || dinfo_init(dev) != 0) return OSCAR_ERR_LAUNCH;
  const bool big = a.g.G > 4;
  switch (a.g.D) {
    case 128: return big ? launch_decode_d<128, 2>(a, stream) : launch_decode_d<128, 1>(a, stream);
    case 256: return big ? launch_decode_d<256, 2>(a, stream) : launch_decode_d<256, 1>(a, stream);
    case 512: return big ? launch_decode_d<512, 2>(a, stream) : launch_decode_d<512, 1>(a, stream);
    default: return OSCAR_ERR_UNSUPPORTED;
  }
}

}  // namespace oscar
