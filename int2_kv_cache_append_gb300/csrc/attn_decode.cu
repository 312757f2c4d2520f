// attn_decode: one decode step of attention over the mixed INT2 / BF16 cache.
//
// Source: hysenlabs article on FutureMLS-Lab/OSCAR (How the offline rotation
// is fit: a fused mixed-precision flash attention over the INT2 + BF16 layout,
// no dequantise-then-attend pass); "OSCAR-LLAMACPP-Gemma-4-12B-it-INT2-KV"
// card (Folders: the rotation applies to Q/K and V); "OSCAR-RotationZoo" (How
// to use: V rotation absorbed into the output).
//
// Two kernels per call (three at head_dim 256/512 with V un-rotated, see unrot):
//   qrot   q' = q R_K * sm_scale * log2(e) (float32; with the in-quant
//          Hadamard a warp transform instead of R_K) written as the split
//          kernel's ready mma fragments, with per-group sums of q'; zeroes the
//          merge tickets and writes the output of empty sequences.
//   split  a persistent grid of P CTAs (by default as many as are resident at
//          once).  The block lists of all (sequence, KV head) units, in unit
//          order, are concatenated and cut by time-weighted block costs into P
//          equal slices, one per CTA, so every CTA has the same amount of work
//          and the grid ends in one wave.  With V kept BF16 (K-only INT2, a
//          separate instantiation) the INT2 part of a unit is cut into 16-token
//          blocks of INT2 K codes with BF16 V rows.  A slice covers the tail of one unit, whole
//          units and the head of another; each such unit part is a segment.
//          Four warps form teams (one warp per 128-channel quant group); each
//          team issues the bulk copies of its own blocks (cp.async.bulk for
//          128-token INT2 blocks: codes + scale/zero; 2-D TMA tensor loads for
//          16-token BF16 sink/ring blocks) into its private stages, running
//          ahead across segment boundaries, and consumes them with mma.sync
//          m16n8k16 in "swap-AB" form: tokens (QK) or channels (PV) on the M
//          side, query heads on N, with each head's hi and lo parts of q' / P
//          in adjacent columns so that the products keep ~22 bits.  INT2 codes
//          go from shared memory into A fragments with one AND per register
//          (fp16 subnormals, see unpack16); per-token scale/zero are applied
//          algebraically:
//            s_t = scale_t * (q'.c_t) + zero_t * sum(q'),
//            o  += (p_t * scale_t) . c_t  and  zeta += p_t * zero_t.
//          Online softmax in log2 units; for D > 128 the warps of a team split
//          a block's channels by quant group and exchange partial scores.  At
//          the end of a segment the CTA merges its teams and writes one partial
//          (m, l, o') per head into the segment's slot; the last CTA of a unit
//          to finish (an atomic ticket, never a wait) merges the unit's slots
//          by log-sum-exp in one online pass, applies o = o' R_V^T (o' H with
//          the in-quant Hadamard; skipped when absorbed) and stores the
//          bf16/fp32 output and lse.
//   unrot  head_dim 256 / 512, V un-rotated by R_V: o = o' R_V^T for every
//          (sequence, query head) at once, from the merged o' the split
//          kernel leaves in workspace slot 0.
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

// Is o = o' R_V^T applied by unrot_kernel after the split kernel (the merging
// CTA then leaves o' in workspace slot 0)?  At head_dim 256 / 512 always (one
// CTA per unit would read all of R_V through L2); at head_dim 128 when G > 4
// heads share a KV head and there are few units (every unit is then shared by
// tens of CTAs and all merge at the very end, where the 8-head un-rotation is
// ~40 % of the merge).
constexpr int kFewUnits = 16;
__host__ __device__ inline bool unrot_separate(const Geom& g, bool absorb_v, bool hadamard) {
  return !absorb_v && !hadamard && (g.D >= 256 || (g.G > 4 && g.B * g.Hkv <= kFewUnits));
}
constexpr int kSub = 64;                   // tokens per INT2 compute sub-block
constexpr int kBfTok = 16;                 // tokens per BF16 block
constexpr int kMaxSeg = 48;                // segments (units) one window of a CTA's slice lists

template <int D, int NQT>
struct DecCfg {
  static constexpr int Dg = D / kGroup;
  static constexpr int TS = Dg;              // warps per team (one quant group each)
  static constexpr int NTEAMS = kNCW / TS;
  static constexpr int ROWB = D / 4;         // code bytes per token
  // INT2 code rows of 64 or 128 bytes arrive as swizzled TMA boxes: plain
  // rows put the 8 token rows of a code load in the same banks (4- to 8-way
  // conflicts); 32-byte rows (head_dim 128) have none worth a second map
  static constexpr bool SWZ = D >= 256;
  static constexpr int BOXES = D / 64;       // 16-row x 64-column TMA boxes per BF16 matrix
  static constexpr int BOX_BYTES = kBfTok * 128;
  static constexpr int I2_BYTES = kI2Tok * (2 * ROWB + 2 * Dg * 4);
  static constexpr int BF_BYTES = 2 * BOXES * BOX_BYTES;
  static constexpr int STAGE = ((I2_BYTES > BF_BYTES ? I2_BYTES : BF_BYTES) + 1023) / 1024 * 1024;
  // K-only INT2 block (V kept BF16): 16 rows of K codes, their scale/zero,
  // then the V rows as BF16 boxes (1 KB aligned for the 128-byte swizzle)
  static constexpr int VB_SZ = kBfTok * ROWB;
  static constexpr int VB_V = (kBfTok * ROWB + kBfTok * Dg * 4 + 1023) / 1024 * 1024;
  static_assert(VB_V + BOXES * BOX_BYTES <= STAGE, "a K-only INT2 block fits a stage");
  // Each team owns NSTW private stages: it issues the bulk copies of its own
  // blocks into them and consumes them in order, so a stage's barrier phases
  // are produced and awaited by one team only.
  static constexpr int NST = 2 * NTEAMS;  // two stages per team: with them two CTAs fit per SM
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
  // and max/sum [2][head]
  static constexpr int PART_A = NTEAMS * HEADS * (D + 2);
  static constexpr int PART_B = HEADS * (D + 2);
  static constexpr int PART_BYTES = (PART_A > PART_B ? PART_A : PART_B) * 4;
  static constexpr int OFF_SEG = OFF_PART + PART_BYTES;             // segment table of a window
  static constexpr int OFF_BAR = OFF_SEG + kMaxSeg * 64;
  static constexpr int SMEM = OFF_BAR + (NST + 2) * 8 + 16 + 1024;  // + slack to align the base to 1 KB
  static_assert(SMEM + 2 * 1024 + 64 <= 227 * 1024, "dynamic + static shared memory of one CTA");
};

// Per-(b, kv head) region sizes and the block list
struct Regions {
  int T, n_sink, tq, n_int, n_ring;
  int ra, rlen1, nrb1;  // ring: first slot, positions before the slot wrap, their blocks
  int nsb, nib, nrb;
  int64_t cbf, ci2;
};

__host__ __device__ inline int imin(int x, int y) { return x < y ? x : y; }
__host__ __device__ inline int imax(int x, int y) { return x > y ? x : y; }

// vb: V kept BF16 at every position; INT2 blocks then hold 16 tokens of INT2
// K codes and BF16 V rows, and weigh like a BF16 block.
__host__ __device__ inline Regions make_regions(int T, int S, int W, int D, int vb, int lm = 0) {
  Regions r;
  r.T = T;
  if (T <= S) {
    r.n_sink = T; r.tq = T; r.n_int = 0; r.n_ring = 0;
  } else {
    r.n_sink = S;
    r.tq = imax(S, T - W);
    r.n_int = r.tq - S;
    r.n_ring = T - r.tq;
  }
  r.nsb = (r.n_sink + kBfTok - 1) / kBfTok;
  static_assert(kI2Tok == 128 && kBfTok == 16, "block counts below are shifts");
  r.nib = vb ? (r.n_int + 15) >> 4 : (r.n_int + 127) >> 7;  // shifts: this runs in every plan pass
  // ring positions [tq, T) sit in slots p mod W: cut them where the slots wrap
  // so that every block reads consecutive slots
  r.ra = r.n_ring > 0 ? r.tq % W : 0;
  r.rlen1 = r.n_ring > 0 ? imin(r.n_ring, W - r.ra) : 0;
  r.nrb1 = (r.rlen1 + kBfTok - 1) / kBfTok;
  r.nrb = r.nrb1 + (r.n_ring - r.rlen1 + kBfTok - 1) / kBfTok;
  // work weights of one block, in proportion to its measured processing time
  // (a 128-token INT2 block takes ~1.8x a 16-token BF16 block for ~1.1x the
  // bytes: the codes are unpacked and the scale/zero algebra is extra work;
  // INT2 weights of 9, 10, 11, 12 and 13 x D timed on the qwen3-4b layer and
  // at head_dim 512: 11 is the best for both; with Lloyd-Max levels every
  // INT2 product runs a second time over the codes' high bits, ~1.7x again:
  // split kernel 61.4 -> 85.5 us on the qwen3-4b layer at 10 and 17)
  r.cbf = int64_t(6) * D;
  r.ci2 = vb ? r.cbf : int64_t(lm ? 17 : 11) * D;
  return r;
}

// Work of one (sequence, KV head) unit of context length T: the summed
// weights of its block list.
__host__ __device__ inline int64_t unit_cost(const Regions& r) {
  return r.nsb * r.cbf + r.nib * r.ci2 + r.nrb * r.cbf;
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
// Work plan of the split kernel.  Units u = b * Hkv + h in order; unit u costs
// unit_cost(T_b) bytes and starts at the sum of the costs before it.  Slice c
// of P is [cut(c), cut(c + 1)).  Normally cut(c) = ceil(c W / P) (W = total);
// a unit [us, ue) is then shared by CTAs floor(us P / W) .. floor((ue-1) P / W),
// and CTA c writes the partial of its segment into slot c - floor(us P / W).
// P is capped so that no unit is shared by more CTAs than the workspace has
// slots.  With fewer than 3 slots the cuts fall on unit boundaries instead
// (cut(c) = start of unit ceil(c U / P)), so every unit has one CTA and slot 0.
// Every CTA computes the same plan from seq_lens; warp-wide loops over B.
// ---------------------------------------------------------------------------
struct Plan {
  int64_t W;     // total cost
  int P;         // CTAs with a slice
  bool aligned;  // cuts on unit boundaries
};

struct SegD {      // one segment: a unit's part of a CTA's slice
  int b, h;        // unit
  int kb, ke;      // block range within the unit's block list
  int slot, nseg;  // partial slot of this CTA, CTAs sharing the unit
  // the unit's block list (the fields of Regions that block_of reads)
  int n_sink, n_int, n_ring, nsb, nib, ra, rlen1, nrb1;
  int pad0, pad1;
};

// block_at on a segment's copy of its unit's block list (VB: 16-token
// INT2 blocks of the K-only INT2 cache)
template <bool VB>
__device__ __forceinline__ Blk block_of(const SegD& r, int k) {
  constexpr int I2T = VB ? kBfTok : kI2Tok;
  Blk b;
  if (k < r.nsb) {
    b.type = 0; b.first = k * kBfTok; b.count = min(kBfTok, r.n_sink - b.first);
  } else if (k < r.nsb + r.nib) {
    b.type = 1; b.first = (k - r.nsb) * I2T; b.count = min(I2T, r.n_int - b.first);
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

// Position of ring slot `slot` of a segment's unit: the ring holds positions
// [tq, T) in slots p mod W, cut into the run from slot ra and the wrapped run
// from slot 0.
__device__ __forceinline__ int ring_pos(const SegD& r, int slot) {
  const int tq = r.n_sink + r.n_int;
  return slot >= r.ra ? tq + slot - r.ra : tq + r.rlen1 + slot;
}

// 2^e as a float, for -126 <= e <= 127
__device__ __forceinline__ float pow2f(int e) { return __int_as_float((e + 127) << 23); }

// the e with x < 2^e <= 2x for finite x > 0 (frexpf's exponent; -126 below the normal range)
__device__ __forceinline__ int exp_above(float x) {
  const int E = (__float_as_int(x) >> 23) & 255;
  return E == 0 ? -126 : E - 126;
}

// floor(x / d) for 0 <= x < 2^62, 0 < d: three fp32 reciprocal estimates and an
// exact int64 correction (FP64 and 64-bit integer division are long software
// sequences on this GPU; this is a few instructions)
__device__ __forceinline__ int64_t div_floor(int64_t x, int64_t d) {
  const float inv = 1.0f / float(d);
  int64_t q = int64_t(float(x) * inv);
  int64_t r = x - q * d;
  q += int64_t(floorf(float(r) * inv));  // each step leaves ~22 fewer bits of error
  r = x - q * d;
  q += int64_t(floorf(float(r) * inv));
  r = x - q * d;
  while (r < 0) { --q; r += d; }
  while (r >= d) { ++q; r -= d; }
  return q;
}

// clamped context lengths of the first kLenCache sequences, staged in shared
// memory once per CTA; the rest are read from global memory
constexpr int kLenCache = 512;
__device__ __forceinline__ int seq_len_at(const DecodeArgs& a, const int* lens, int b) {
  return b < kLenCache ? lens[b] : clamp_seq_len(a, b);
}

// floor(x / d) when the quotient is known to be below 2^20 (one fp32 estimate,
// off by at most one, then corrected exactly)
__device__ __forceinline__ int64_t div_small(int64_t x, int64_t d) {
  int64_t q = int64_t(float(x) * (1.0f / float(d)));
  int64_t r = x - q * d;
  while (r < 0) { --q; r += d; }
  while (r >= d) { ++q; r -= d; }
  return q;
}

template <int D, bool VB, bool LM>
__device__ __forceinline__ int64_t seq_cost(const DecodeArgs& a, const int* lens, int b) {
  return b < a.g.B ? unit_cost(make_regions(seq_len_at(a, lens, b), a.g.S, a.g.W, D, VB, LM)) : 0;
}

template <int D, bool VB, bool LM>
__device__ Plan make_plan(const DecodeArgs& a, const int* lens, int lane) {
  const Geom& g = a.g;
  int64_t W = 0, cmax = 0;
  for (int b0 = 0; b0 < g.B; b0 += 32) {
    int64_t sm = seq_cost<D, VB, LM>(a, lens, b0 + lane), mx = sm;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      sm += __shfl_xor_sync(0xffffffffu, sm, o);
      mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    }
    W += sm * g.Hkv;
    cmax = max(cmax, mx);
  }
  Plan pl;
  pl.W = W;
  pl.aligned = a.ns < 3;
  int64_t P = gridDim.x;
  if (pl.aligned) {
    P = min(P, int64_t(g.B) * g.Hkv);
  } else if (W > 0) {
    P = min(P, W);
    P = min(P, max(int64_t(1), div_floor((int64_t(a.ns) - 2) * W, cmax)));
  }
  pl.P = int(max(P, int64_t(1)));
  return pl;
}

// Start cost of unit k (k <= B * Hkv).
template <int D, bool VB, bool LM>
__device__ int64_t unit_start(const DecodeArgs& a, const int* lens, int lane, int64_t k) {
  const int Hkv = a.g.Hkv;
  const int bk = int(k) / Hkv, hk = int(k) % Hkv;  // k <= B * Hkv < 2^31
  int64_t base = 0;
  for (int b0 = 0; b0 < bk; b0 += 32) {
    int64_t c = b0 + lane < bk ? seq_cost<D, VB, LM>(a, lens, b0 + lane) * Hkv : 0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
    base += c;
  }
  return base + (hk > 0 ? hk * seq_cost<D, VB, LM>(a, lens, bk) : 0);
}

// Unit holding cost x (0 <= x < W) and its start cost.
template <int D, bool VB, bool LM>
__device__ void locate(const DecodeArgs& a, const int* lens, int lane, int64_t x, int& u, int64_t& us) {
  const int Hkv = a.g.Hkv;
  int64_t base = 0;
  u = 0;
  us = 0;
  for (int b0 = 0; b0 < a.g.B; b0 += 32) {
    const int64_t per = seq_cost<D, VB, LM>(a, lens, b0 + lane);
    int64_t incl = per * Hkv;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    const unsigned hit = __ballot_sync(0xffffffffu, base + incl > x);
    if (hit) {
      const int l = __ffs(hit) - 1;
      const int64_t pre = base + __shfl_sync(0xffffffffu, incl, l) - __shfl_sync(0xffffffffu, per, l) * Hkv;
      const int64_t pl = __shfl_sync(0xffffffffu, per, l);
      const int h = int(div_small(x - pre, pl));  // h < Hkv
      u = (b0 + l) * Hkv + h;
      us = pre + int64_t(h) * pl;
      return;
    }
    base += __shfl_sync(0xffffffffu, incl, 31);
  }
}

// Segment table of one window of slice [lo, hi) of CTA c, from unit u with
// start cost us (warp-wide; lane 0's results are the ones used).  Lists at most
// kMaxSeg segments; returns their number and leaves (u, us) at the first unit
// not listed.
template <int D, bool VB, bool LM>
__device__ int build_segments(const DecodeArgs& a, const int* lens, const Plan& pl, int c, int64_t lo, int64_t hi,
                              int& u, int64_t& us, SegD* seg, int lane) {
  const Geom& g = a.g;
  const int64_t U = int64_t(g.B) * g.Hkv;
  int n = 0;
  while (us < hi && u < U && n < kMaxSeg) {
    const int64_t uu = u + lane;
    const int b = int(uu) / g.Hkv, h = int(uu) % g.Hkv;
    const int T = uu < U ? seq_len_at(a, lens, b) : 0;
    const Regions rg = make_regions(T, g.S, g.W, D, VB, LM);
    const int64_t cu = uu < U ? unit_cost(rg) : 0;
    int64_t incl = cu;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    const int64_t s0 = us + incl - cu, e0 = us + incl;
    const bool take = cu > 0 && s0 < hi;
    const unsigned tk = __ballot_sync(0xffffffffu, take);
    const int idx = n + __popc(tk & ((1u << lane) - 1u));
    if (take && idx < kMaxSeg) {
      SegD d;
      d.b = b; d.h = h;
      d.n_sink = rg.n_sink; d.n_int = rg.n_int; d.n_ring = rg.n_ring;
      d.nsb = rg.nsb; d.nib = rg.nib; d.ra = rg.ra; d.rlen1 = rg.rlen1; d.nrb1 = rg.nrb1;
      d.pad0 = 0; d.pad1 = 0;
      d.kb = first_block_at(rg, max(lo, s0) - s0);
      d.ke = first_block_at(rg, min(hi, e0) - s0);
      if (pl.aligned) {
        d.slot = 0; d.nseg = 1;
      } else {
        const int64_t cf = div_small(s0 * pl.P, pl.W), cl = div_small((e0 - 1) * pl.P, pl.W);  // < P
        d.slot = int(c - cf);
        d.nseg = int(cl - cf + 1);
      }
      seg[idx] = d;
    }
    // advance past the units listed (or skipped), stopping at a full table
    const int room = kMaxSeg - n;
    int adv = 32;
    if (__popc(tk) > room) {
      // the (room+1)-th taken lane is the first unit not listed
      unsigned m = tk;
      for (int i = 0; i < room; ++i) m &= m - 1;
      adv = __ffs(m) - 1;
    }
    const int64_t consumed = adv > 0 ? __shfl_sync(0xffffffffu, incl, adv - 1) : 0;
    n += min(__popc(tk), room);
    us += consumed;
    u += adv;
  }
  return n;
}

// ---------------------------------------------------------------------------
// qrot: q' = q R_K * qscale for the G query heads of one (b, kv head) and one
// 128-channel quant group, written as the split kernel's mma B fragments (see
// the two layouts below) with per-group sums and score factors; the group-0
// CTA also zeroes that unit's merge ticket.  For an empty sequence it writes the output
// instead (zeros, lse = -inf) and flags OSCAR_DEV_EMPTY.  512 threads = 4 slices of the contraction index
// x 128 output columns, so each thread has at most D/4 loads of R_K, issued
// 32 at a time.  Launched with PDL: it waits for the preceding kernel before
// reading anything (q may be produced right before this call) and then at
// once lets the split kernel launch, whose CTAs start their cache copies
// while this kernel computes; the split kernel reads q' only after its own
// wait for this grid's completion.  In decode_step it computes while the
// append runs and waits for the append only before exiting.
// ---------------------------------------------------------------------------
constexpr int kQrotThreads = 512;

template <int D>
__global__ void __launch_bounds__(kQrotThreads) qrot_kernel(const DecodeArgs a) {
  constexpr int KP = kQrotThreads / 128;  // slices of the contraction index
  constexpr int KC = D / KP;              // contraction indices per slice
  __shared__ float qs[8][D];
  __shared__ float part[KP - 1][8][128];
  __shared__ float qv[8][128];  // q' of this group, per head
  __shared__ float red[8][4], redm[8][4];
  __shared__ int Xs[8];
  const int bh = blockIdx.x;  // b * Hkv + h
  const int chunk = blockIdx.y;
  const int G = a.g.G;
  const int c = threadIdx.x & 127, kp = threadIdx.x >> 7;
  const int col = chunk * 128 + c;
  const int64_t q0 = int64_t(bh) * G * D;  // first query head of this kv head
  // In a fused step (decode_step) the split kernel may launch at once (it only
  // streams cache blocks the preceding append leaves untouched before waiting
  // for this grid), and this grid does not wait for the append before working:
  // it reads only q, R_K and seq_lens, complete before the call's append began.
  // It waits for the append just before exiting, so that its completion, which
  // the split kernel waits for, still implies the append's.  Otherwise it waits
  // first (q may be produced right before this call) and then lets the split
  // kernel launch.
  if (a.fused) {
    pdl_trigger();
  } else {
    pdl_wait();
    pdl_trigger();
  }

  const int b = bh / a.g.Hkv;
  const int T = clamp_seq_len(a, b);
  if (chunk == 0 && threadIdx.x == 0 && bh % a.g.Hkv == 0) {
    if (a.seq_lens[b] > a.g.cap) status_or(a.status, OSCAR_DEV_OVER_CAPACITY);
    if (T < 1) status_or(a.status, OSCAR_DEV_EMPTY);
  }
  if (T < 1) {
    // nothing to attend to (the split kernel has no work here): zero output, lse = -inf
    for (int idx = threadIdx.x; idx < G * 128; idx += kQrotThreads) {
      const int64_t oi = q0 + int64_t(idx / 128) * D + chunk * 128 + idx % 128;
      if (a.out_fp32)
        static_cast<float*>(a.out)[oi] = 0.f;
      else
        static_cast<__nv_bfloat16*>(a.out)[oi] = __float2bfloat16_rn(0.f);
    }
    if (chunk == 0 && threadIdx.x < G && a.lse) a.lse[q0 / D + threadIdx.x] = -INFINITY;
    if (a.fused) pdl_wait();
    return;
  }

  // column c of this group before scaling: q R_K, or the in-quant Hadamard
  // transform of the group (warp i transforms head i)
  float hsum[8];
  if (a.hadamard) {
    const int w = threadIdx.x >> 5, ln = threadIdx.x & 31;
    if (w < G) {
      float x[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int64_t qi = q0 + int64_t(w) * D + chunk * 128 + ln + 32 * e;
        x[e] = a.in_fp32 ? static_cast<const float*>(a.q)[qi]
                         : __bfloat162float(static_cast<const __nv_bfloat16*>(a.q)[qi]);
      }
      hadamard128_warp(x, ln);
#pragma unroll
      for (int e = 0; e < 4; ++e) qv[w][ln + 32 * e] = x[e];
    }
    if (chunk == 0 && threadIdx.x == 0) a.ticket[bh] = 0;
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 8; ++i) hsum[i] = (kp == 0 && i < G) ? qv[i][c] : 0.f;
  } else {
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
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      hsum[i] = 0.f;
      if (kp == 0 && i < G) {
        float sum = acc[i];
#pragma unroll
        for (int p = 0; p < KP - 1; ++p) sum += part[p][i][c];
        hsum[i] = sum;
      }
    }
  }
  if (kp == 0) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (i < G) {
        const float sum = hsum[i];
        const float v = sum * a.qscale;
        if (!(fabsf(v) < 60000.f)) status_or(a.status, OSCAR_DEV_FP16_RANGE);
        qv[i][c] = v;
        float t = v, m = fabsf(v);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          t += __shfl_xor_sync(0xffffffffu, t, o);
          m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        }
        if ((c & 31) == 0) {
          red[i][c >> 5] = t;
          redm[i][c >> 5] = m;
        }
      }
    }
  }
  __syncthreads();
  // per head: sum of q' over the group, and the exponent X that puts the
  // largest |q'| * 2^X in [2^13, 2^14) (the INT2 fragments are scaled by it)
  if (threadIdx.x < G) {
    const int i = threadIdx.x;
    const float mx = fmaxf(fmaxf(redm[i][0], redm[i][1]), fmaxf(redm[i][2], redm[i][3]));
    const int X = mx > 0.f ? max(-100, min(14 - exp_above(mx), 100)) : 0;
    Xs[i] = X;
    const int64_t qi = (q0 / D + i) * (D / kGroup) + chunk;
    a.qsum[qi] = red[i][0] + red[i][1] + red[i][2] + red[i][3];
    a.qF[qi] = pow2f(24 - X);
  }
  __syncthreads();

  // B fragments of this (b, kv head, group) for the split kernel's mma.sync
  // m16n8k16, in its lanes' order.  Column n of an n-tile nq is head slot
  // 4 nq + n / 2, with the hi (n even) or lo (n odd) part; lane = 4 gq + cq
  // holds column gq and k-rows 2cq, 2cq + 1 (+ 8 for the second register).
  const int NQT = G > 4 ? 2 : 1, NQB = 2 * NQT;
  const int64_t grp = int64_t(bh) * (D / kGroup) + chunk;
  // INT2 blocks: channel d of a K code at mantissa bit 2k meets q'[d] * 4^-k * 2^X
  // as an fp16 hi/lo pair (k = unpack_kq of its register, see unpack16), entry
  // ((nq * 8 + kk) * 2 + half) * 32 + lane
  for (int e = threadIdx.x; e < NQT * 512; e += kQrotThreads) {
    const int ln = e & 31, half = (e >> 5) & 1, kk = (e >> 6) & 7, nq = e >> 9;
    const int gq = ln >> 2, cq = ln & 3, hb = 4 * nq + (gq >> 1);
    const int d0 = 16 * kk + 2 * cq + 8 * half;
    uint32_t v16 = 0;
    if (hb < G) {
      const float f = pow2f(Xs[hb] - 2 * unpack_kq(2 * (kk & 3) + half));
      const uint32_t s0 = split_f16(qv[hb][d0] * f), s1 = split_f16(qv[hb][d0 + 1] * f);
      v16 = (gq & 1) ? ((s0 >> 16) | (s1 & 0xffff0000u)) : ((s0 & 0xffffu) | (s1 << 16));
    }
    a.qfrag[grp * (NQT * 512) + e] = v16;
  }
  // BF16 blocks: n-tile 2nq holds the (hi, mid) and n-tile 2nq + 1 the (lo, 0)
  // parts of each head's three-way bf16 split of q' (~24 bits), entry
  // ((kk * NQB + nb) * 2 + half) * 32 + lane: the split kernel's shared image
  for (int e = threadIdx.x; e < NQT * 1024; e += kQrotThreads) {
    const int ln = e & 31, half = (e >> 5) & 1, nb = (e >> 6) % NQB, kk = (e >> 6) / NQB;
    const int gq = ln >> 2, cq = ln & 3, hb = 4 * (nb >> 1) + (gq >> 1);
    const int d0 = 16 * kk + 2 * cq + 8 * half;
    uint32_t w = 0;
    if (hb < G) {
      uint32_t p0[3], p1[3];
      split3_bf16(qv[hb][d0], p0);
      split3_bf16(qv[hb][d0 + 1], p1);
      if (nb & 1)
        w = (gq & 1) ? 0u : (p0[2] | (p1[2] << 16));
      else
        w = (gq & 1) ? (p0[1] | (p1[1] << 16)) : (p0[0] | (p1[0] << 16));
    }
    a.qbfrag[grp * (NQT * 1024) + e] = w;
  }
  if (a.fused) pdl_wait();  // see above: completion implies the append's
}

// ---------------------------------------------------------------------------
// split kernel
// ---------------------------------------------------------------------------
// VB: the cache keeps V as BF16 at every position (K-only INT2); LM: INT2
// codes index the Lloyd-Max levels, level(c) = rho * c + kLmHi * (2 c1), so each
// INT2 product runs a second time over the codes' high bits.  Separate
// instantiations: the default kernel carries none of either mode's code.
// XOR applied by the TMA swizzle (32, 64 or 128 bytes, the code row size
// ROWB) to the 16-byte chunk index of token row t of a stage's code matrix:
// address bits 7.. of the row start, masked to the chunk-index bits.
template <int ROWB>
__device__ __forceinline__ uint32_t code_chunk_xor(int t) {
  return (uint32_t(t * ROWB) >> 7) & uint32_t(ROWB / 16 - 1);
}

template <int D, int NQT, bool VB, bool LM>
__global__ void __launch_bounds__(kThreads, 2)
    split_kernel(const __grid_constant__ CUtensorMap tks, const __grid_constant__ CUtensorMap tvs,
                 const __grid_constant__ CUtensorMap tkr, const __grid_constant__ CUtensorMap tvr,
                 const __grid_constant__ CUtensorMap tkc, const __grid_constant__ CUtensorMap tvc,
                 const DecodeArgs a) {
  using C = DecCfg<D, NQT>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 128-byte-swizzled TMA destinations need 1 KB alignment
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  SegD* seg = reinterpret_cast<SegD*>(smem + C::OFF_SEG);
  __shared__ int abort_flag, is_last, win_n, win_more;

  __shared__ int lens[kLenCache];

  const Geom& g = a.g;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < g.B && i < kLenCache; i += kThreads) lens[i] = clamp_seq_len(a, i);
  __syncthreads();

  // ---- this CTA's slice [lo, hi) of the concatenated unit costs
  const Plan pl = make_plan<D, VB, LM>(a, lens, lane);
  const int c = blockIdx.x;
  if (pl.W == 0 || c >= pl.P) return;
  int64_t lo, hi, us_next = 0;
  int u_next = 0;
  if (pl.aligned) {
    const int64_t U = int64_t(g.B) * g.Hkv;
    const int64_t k0 = div_floor(int64_t(c) * U + pl.P - 1, pl.P), k1 = div_floor(int64_t(c + 1) * U + pl.P - 1, pl.P);
    lo = unit_start<D, VB, LM>(a, lens, lane, k0);
    hi = unit_start<D, VB, LM>(a, lens, lane, k1);
    u_next = int(k0);
    us_next = lo;
  } else {
    lo = div_floor(int64_t(c) * pl.W + pl.P - 1, pl.P);
    hi = div_floor(int64_t(c + 1) * pl.W + pl.P - 1, pl.P);
    if (lo < hi) locate<D, VB, LM>(a, lens, lane, lo, u_next, us_next);
  }
  if (lo >= hi) return;

  if (!a.fused) pdl_wait();  // q' and the merge tickets come from the preceding kernel

  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int s = 0; s < C::NST; ++s) mbar_init(smem_u32(&bars[s]), 1);  // issuer's arrival + tx bytes
    mbar_init(smem_u32(&bars[C::NST]), 1);      // R_V prefetch of a merge in the last segment
    mbar_init(smem_u32(&bars[C::NST + 1]), 1);  // shared bf16 q' fragments
    mbar_fence_init();
  }

  const uint8_t* kbase = a.layer_base;
  const uint8_t* vbase = a.layer_base + g.role_bytes;
  const uint64_t codes_off = g.sink_bytes + g.ring_bytes;
  const uint64_t sz_off = codes_off + g.codes_bytes;

  const int team = warp / C::TS, wt = warp % C::TS;  // wt = quant group handled
  const int gq = lane >> 2, cq = lane & 3;
  // Columns of this lane's INT2 code loads in a 128-token stage: K bytes
  // 32 wt + 8 cq of rows 16 m + gq (+ 8), V word 8 wt + gq of rows
  // 16 k + 2 cq + {0, 1} (+ 8).  In the swizzled stage (head_dim >= 256) the
  // 16-byte chunk c of token row t sits at chunk c ^ code_chunk_xor(t), an XOR
  // that depends only on t mod 8, which the lane fixes.
  const int kcol = C::SWZ ? int(((uint32_t(2 * wt + (cq >> 1)) ^ code_chunk_xor<C::ROWB>(gq)) << 4) |
                                uint32_t(8 * (cq & 1)))
                          : wt * 32 + cq * 8;
  const int vcol0 = C::SWZ ? int(((uint32_t(2 * wt + (gq >> 2)) ^ code_chunk_xor<C::ROWB>(2 * cq)) << 2) |
                                 uint32_t(gq & 3))
                           : wt * 8 + gq;
  const int vcol1 = C::SWZ ? int(((uint32_t(2 * wt + (gq >> 2)) ^ code_chunk_xor<C::ROWB>(2 * cq + 1)) << 2) |
                                 uint32_t(gq & 3))
                           : wt * 8 + gq;
  const int Gh = g.G;
  auto my_stage = [&](int j) { return team * C::NSTW + j % C::NSTW; };
  int issued = 0, consumed = 0;  // blocks of this team issued / consumed so far
  int is_ = 0, ij = 0;           // issue cursor: segment, team-local block index
  int nwin = 0;                  // segments in the current window

  // Bulk copies of block k of segment si into stage `stage`, issued by the
  // calling warp (lane 0 arms the barrier with the byte count first).
  auto issue_block = [&](int si, int k, int stage) {
    const SegD& sd = seg[si];
    const Blk bk = block_of<VB>(sd, k);
    const int64_t bh = int64_t(sd.b) * g.Hkv + sd.h;
    const uint32_t full = smem_u32(&bars[stage]);
    const uint32_t dst = smem_u32(smem + C::OFF_STAGE + stage * C::STAGE);
    // test hook: CTA 0's first block expects bytes no copy delivers, so its
    // wait runs out (every copy issued still completes)
    const uint32_t extra = (a.wait_poison > 0 && blockIdx.x == 0 && issued == 0 && team == 0) ? a.wait_poison : 0;
    if (bk.type == 1) {
      if (lane == 0) {
        const int n4 = (bk.count + 3) & ~3;
        const uint32_t cb = n4 * C::ROWB, sb = n4 * C::Dg * 4;
        const int64_t row = bh * g.ncap + bk.first;
        if constexpr (VB) {
          // K codes and scale/zero, and the BF16 V rows of the same positions
          mbar_arrive_expect_tx(full, cb + sb + C::BOXES * C::BOX_BYTES + extra);
          bulk_g2s(dst, kbase + codes_off + row * C::ROWB, cb, full);
          bulk_g2s(dst + C::VB_SZ, kbase + sz_off + row * C::Dg * 4, sb, full);
          const int vrow = int(bh * g.cap + g.S + bk.first);
#pragma unroll
          for (int q = 0; q < C::BOXES; ++q) tma_load_2d(dst + C::VB_V + q * C::BOX_BYTES, &tvs, 64 * q, vrow, full);
        } else if constexpr (C::SWZ) {
          // K and V codes as 128-row TMA boxes, swizzled by the row size (see
          // code_chunk_xor); rows past the unit's last token are not used
          mbar_arrive_expect_tx(full, 2 * kI2Tok * C::ROWB + 2 * sb + extra);
          tma_load_2d(dst, &tkc, 0, int(row), full);
          tma_load_2d(dst + kI2Tok * C::ROWB, &tvc, 0, int(row), full);
          bulk_g2s(dst + 2 * kI2Tok * C::ROWB, kbase + sz_off + row * C::Dg * 4, sb, full);
          bulk_g2s(dst + 2 * kI2Tok * C::ROWB + kI2Tok * C::Dg * 4, vbase + sz_off + row * C::Dg * 4, sb, full);
        } else {
          mbar_arrive_expect_tx(full, 2 * cb + 2 * sb + extra);
          bulk_g2s(dst, kbase + codes_off + row * C::ROWB, cb, full);
          bulk_g2s(dst + kI2Tok * C::ROWB, vbase + codes_off + row * C::ROWB, cb, full);
          bulk_g2s(dst + 2 * kI2Tok * C::ROWB, kbase + sz_off + row * C::Dg * 4, sb, full);
          bulk_g2s(dst + 2 * kI2Tok * C::ROWB + kI2Tok * C::Dg * 4, vbase + sz_off + row * C::Dg * 4, sb, full);
        }
      }
    } else {
      // 16 rows of K and V as 64-column boxes, 128-byte swizzled by the TMA unit
      // (with V kept BF16, V rows come from the position-indexed V map)
      if (lane == 0) {
        mbar_arrive_expect_tx(full, 2 * C::BOXES * C::BOX_BYTES + extra);
        const CUtensorMap* mk = bk.type == 0 ? &tks : &tkr;
        const CUtensorMap* mv = (bk.type == 0 || VB) ? &tvs : &tvr;
        const int row0 = int(bk.type == 0 ? bh * g.S + bk.first : bh * g.W + bk.first);
        const int vrow0 = VB ? int(bh * g.cap + (bk.type == 0 ? bk.first : ring_pos(sd, bk.first))) : row0;
#pragma unroll
        for (int q = 0; q < C::BOXES; ++q) {
          tma_load_2d(dst + q * C::BOX_BYTES, mk, 64 * q, row0, full);
          tma_load_2d(dst + (C::BOXES + q) * C::BOX_BYTES, mv, 64 * q, vrow0, full);
        }
      }
    }
  };

  // In a fused step: does block k of a segment hold a location the preceding
  // append writes (sink positions and INT2 rows of [new_pos, new_pos + new_n),
  // ring slots of its last min(new_n, W) positions)?
  auto written = [&](const SegD& sx, int k) -> bool {
    const Blk bk = block_of<VB>(sx, k);
    const int st = a.new_pos[sx.b], n = a.new_n;
    if (n <= 0) return false;
    if (bk.type == 0) return bk.first < min(st + n, g.S) && st < bk.first + bk.count;
    if (bk.type == 1) {
      const int p0 = g.S + bk.first;
      return p0 < st + n && max(st, g.S) < p0 + bk.count;
    }
    if constexpr (VB) {  // the V rows of a ring block sit at its positions
      const int p0 = ring_pos(sx, bk.first);
      if (p0 < st + n && st < p0 + bk.count) return true;
    }
    const int w0 = max(max(st, st + n - g.W), 0), wn = st + n - w0;  // ring positions written
    if (wn <= 0) return false;
    if (wn >= g.W) return true;
    const int a0 = w0 % g.W;
    return (bk.first - a0 + g.W) % g.W < wn || (a0 - bk.first + g.W) % g.W < bk.count;
  };
  // the team's next block in window order (blocks kb + team + j * NTEAMS of
  // each segment), if any: issue it into the team's next stage (with
  // old_only, not if the preceding append writes it)
  auto issue_next = [&](bool old_only = false) {
    while (is_ < nwin) {
      const int k = seg[is_].kb + team + ij * C::NTEAMS;
      if (k < seg[is_].ke) {
        if (old_only && written(seg[is_], k)) return false;
        issue_block(is_, k, my_stage(issued));
        ++issued;
        ++ij;
        return true;
      }
      ++is_;
      ij = 0;
    }
    return false;
  };

  // q' of a segment's unit, prepared by qrot: this lane's B fragments of group
  // wt (INT2 blocks), and the per-group sums and score factors of the heads of
  // its C fragments (head slot 4 nq + cq)
  auto load_q = [&](int bx, int hx, uint32_t (&qfx)[8][NQT][2], float (&qsx)[NQT], float (&qFx)[NQT]) {
    const int64_t unit = int64_t(bx) * g.Hkv + hx;
    const uint32_t* src = a.qfrag + (unit * C::Dg + wt) * (NQT * 512);
#pragma unroll
    for (int nq = 0; nq < NQT; ++nq) {
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
#pragma unroll
        for (int half = 0; half < 2; ++half) qfx[kk][nq][half] = src[((nq * 8 + kk) * 2 + half) * 32 + lane];
      const int hc = 4 * nq + cq;
      const int64_t qi = (int64_t(bx) * g.Hq + hx * Gh + hc) * C::Dg + wt;
      qsx[nq] = hc < Gh ? a.qsum[qi] : 0.f;
      qFx[nq] = hc < Gh ? a.qF[qi] : 1.f;
    }
  };
  // bf16 fragments of a unit (all its groups) into the shared image, one bulk
  // copy issued by thread 0 on barrier NST + 1; every copy is awaited in order
  const uint32_t qb_bar = smem_u32(&bars[C::NST + 1]);
  int qb_issued = 0, qb_waited = 0;
  auto qb_issue = [&](int bx, int hx) {
    if (threadIdx.x == 0) {
      const int64_t unit = int64_t(bx) * g.Hkv + hx;
      mbar_arrive_expect_tx(qb_bar, C::QBF_BYTES);
      bulk_g2s(smem_u32(smem + C::OFF_QBF), a.qbfrag + unit * (C::Dg * NQT * 1024), C::QBF_BYTES, qb_bar);
    }
    ++qb_issued;
  };
  auto qb_wait = [&]() {  // thread 0 waits; a CTA barrier must follow before others read
    if (threadIdx.x == 0 && !mbar_wait(qb_bar, qb_waited & 1, a.wait_ns)) {
      abort_flag = 1;
      status_or(a.status, OSCAR_DEV_TIMEOUT);
    }
    ++qb_waited;
  };


  // the first window starts at unit u_next: its q' is loaded now, ahead of
  // the window's copies, and lands while the segment table is built
  uint32_t qf[8][NQT][2];
  float qsum[NQT], qF[NQT];
  const int pre_b = u_next / g.Hkv, pre_h = u_next % g.Hkv;
  if (!a.fused) {
    load_q(pre_b, pre_h, qf, qsum, qF);
    qb_issue(pre_b, pre_h);
  }
  bool first = true, aborted = false;
  for (;;) {
    // ---- segment table of the next window (warp 0), then start streaming
    if (warp == 0) {
      const int n = build_segments<D, VB, LM>(a, lens, pl, c, lo, hi, u_next, us_next, seg, lane);
      if (lane == 0) {
        win_n = n;
        win_more = us_next < hi && u_next < int64_t(g.B) * g.Hkv;
      }
    }
    __syncthreads();
    nwin = win_n;
    const bool more = win_more;
    is_ = 0;
    ij = 0;
    if (first && a.fused) {
      // blocks the append leaves alone stream while it and qrot run
      if (wt == 0)
        for (int i = 0; i < C::NSTW; ++i)
          if (!issue_next(true)) break;
      pdl_wait();  // the append, q' and the merge tickets are complete
      if (nwin > 0) {
        load_q(seg[0].b, seg[0].h, qf, qsum, qF);
        qb_issue(seg[0].b, seg[0].h);
      }
      if (wt == 0)
        while (issued < C::NSTW && issue_next()) {
        }
    } else {
      // (with cuts on unit boundaries the first unit listed can follow empty ones)
      if (nwin > 0 && (!first || seg[0].b != pre_b || seg[0].h != pre_h)) {
        load_q(seg[0].b, seg[0].h, qf, qsum, qF);
        if (qb_issued > qb_waited) qb_wait();  // the shared image is rewritten only once landed
        __syncthreads();
        qb_issue(seg[0].b, seg[0].h);
      }
      if (wt == 0)
        for (int i = 0; i < C::NSTW; ++i) issue_next();
    }
    first = false;

    for (int sg = 0; sg < nwin; ++sg) {
      const SegD& sd = seg[sg];
      const int b = sd.b, h = sd.h;
      const int head0 = h * Gh;  // first query head of this kv head
      const int64_t bh = int64_t(b) * g.Hkv + h;
      if (!more && sg == nwin - 1) pdl_trigger();
      if (sg > 0) load_q(b, h, qf, qsum, qF);  // the shared image of this unit was issued at the previous segment's end

      // bf16 fragments for BF16 blocks (shared by the teams): n-tile 2nq holds
      // (hi, mid) and n-tile 2nq+1 holds (lo, 0) of each head's three-way split
      const uint32_t* qbf = reinterpret_cast<const uint32_t*>(smem + C::OFF_QBF) + wt * 8 * C::NQB * 64;
      qb_wait();
      asm volatile("bar.sync 14, %0;" ::"r"(32 * kNCW) : "memory");  // shared bf16 fragments landed
      if (abort_flag) {
        aborted = true;
        break;
      }

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

      // INT2 P.V takes V codes from unpack16: the code of output row r arrives
      // as code * 2^e(r), e(r) = unpack_exp(p) with p = 2 * (mtd % 4) for rows gq
      // and 2 * (mtd % 4) + 1 for rows gq + 8.  While INT2 blocks are consumed, row
      // r of o holds (real value) * 2^e(r); it is converted by exact powers of two
      // at a switch between INT2 and BF16 blocks and at the end.
      bool o_i2 = false;
      auto scale_o = [&](int sign) {  // o *= 2^(sign * e(r)) per row
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          const float f0 = pow2f(sign * unpack_exp(2 * (mt & 3)));
          const float f1 = pow2f(sign * unpack_exp(2 * (mt & 3) + 1));
#pragma unroll
          for (int nq = 0; nq < NQT; ++nq) {
            o[mt][nq][0] *= f0; o[mt][nq][1] *= f0;
            o[mt][nq][2] *= f1; o[mt][nq][3] *= f1;
          }
        }
      };


      const int nb = sd.ke - sd.kb;
      const int nmine = nb > team ? (nb - team + C::NTEAMS - 1) / C::NTEAMS : 0;  // this team's blocks
      for (int j = 0; j < nmine; ++j) {
        const int stage = my_stage(consumed);
        int ok = 1;
        if (lane == 0) ok = mbar_wait(smem_u32(&bars[stage]), (consumed / C::NSTW) & 1, a.wait_ns);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        // the warps of a team must take the same decision: they meet at team barriers below
        if constexpr (C::TS > 1) ok = team_all(ok, 1 + team, 32 * C::TS);
        if (!ok) {
          if (lane == 0) { abort_flag = 1; status_or(a.status, OSCAR_DEV_TIMEOUT); }
          break;
        }
        const Blk bk = block_of<VB>(sd, sd.kb + team + j * C::NTEAMS);
        const uint8_t* st = smem + C::OFF_STAGE + stage * C::STAGE;
        // is_i2: K and V from INT2 codes (128-token block); kv16: K-only INT2
        // block (V kept BF16): 16 tokens of INT2 K codes with BF16 V rows
        const bool is_i2 = bk.type == 1 && !VB;
        const bool kv16 = VB && bk.type == 1;
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
              w[i][0] = *reinterpret_cast<const uint2*>(kc + (tb + t0) * C::ROWB + kcol);
              w[i][1] = *reinterpret_cast<const uint2*>(kc + (tb + t0 + 8) * C::ROWB + kcol);
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
            // Lloyd-Max levels: the same products over the codes' high bits
            float acch[MG][NQT][4];
            if constexpr (LM) {
#pragma unroll
              for (int i = 0; i < MG; ++i)
#pragma unroll
                for (int nq = 0; nq < NQT; ++nq)
#pragma unroll
                  for (int e = 0; e < 4; ++e) acch[i][nq][e] = 0.f;
#pragma unroll
              for (int wi = 0; wi < 2; ++wi) {
                uint32_t r[MG][2][8];
#pragma unroll
                for (int i = 0; i < MG; ++i) {
                  unpack16_hi(wi ? w[i][0].y : w[i][0].x, r[i][0]);
                  unpack16_hi(wi ? w[i][1].y : w[i][1].x, r[i][1]);
                }
#pragma unroll
                for (int k4 = 0; k4 < 4; ++k4) {
                  const int kk = 4 * wi + k4;
#pragma unroll
                  for (int nq = 0; nq < NQT; ++nq)
#pragma unroll
                    for (int i = 0; i < MG; ++i)
                      mma_f16(acch[i][nq], r[i][0][2 * k4], r[i][1][2 * k4], r[i][0][2 * k4 + 1],
                              r[i][1][2 * k4 + 1], qf[kk][nq][0], qf[kk][nq][1]);
                }
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
                if constexpr (LM) {
                  const float d0 = fmaf(kLmRho, acc[i][nq][0] + acc[i][nq][1], kLmHi * (acch[i][nq][0] + acch[i][nq][1]));
                  const float d1 = fmaf(kLmRho, acc[i][nq][2] + acc[i][nq][3], kLmHi * (acch[i][nq][2] + acch[i][nq][3]));
                  s[mt][nq][0] = fmaf(ksc[mt][0], d0 * qF[nq], kze[mt][0] * qsum[nq]);
                  s[mt][nq][1] = fmaf(ksc[mt][1], d1 * qF[nq], kze[mt][1] * qsum[nq]);
                } else {
                  s[mt][nq][0] = fmaf(ksc[mt][0], (acc[i][nq][0] + acc[i][nq][1]) * qF[nq], kze[mt][0] * qsum[nq]);
                  s[mt][nq][1] = fmaf(ksc[mt][1], (acc[i][nq][2] + acc[i][nq][3]) * qF[nq], kze[mt][1] * qsum[nq]);
                }
              }
            }
          }
        } else if (kv16) {
          // one m-tile: the INT2 scores of the 128-token path for tokens gq, gq + 8
          const uint32_t* ksz = reinterpret_cast<const uint32_t*>(st + C::VB_SZ);
          const uint2 w0 = *reinterpret_cast<const uint2*>(st + gq * C::ROWB + wt * 32 + cq * 8);
          const uint2 w1 = *reinterpret_cast<const uint2*>(st + (gq + 8) * C::ROWB + wt * 32 + cq * 8);
          float acc[NQT][4];
#pragma unroll
          for (int nq = 0; nq < NQT; ++nq)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[nq][e] = 0.f;
#pragma unroll
          for (int wi = 0; wi < 2; ++wi) {
            uint32_t r0[8], r1[8];
            unpack16(wi ? w0.y : w0.x, r0);
            unpack16(wi ? w1.y : w1.x, r1);
#pragma unroll
            for (int k4 = 0; k4 < 4; ++k4)
#pragma unroll
              for (int nq = 0; nq < NQT; ++nq)
                mma_f16(acc[nq], r0[2 * k4], r1[2 * k4], r0[2 * k4 + 1], r1[2 * k4 + 1], qf[4 * wi + k4][nq][0],
                        qf[4 * wi + k4][nq][1]);
          }
          float acch[NQT][4];
          if constexpr (LM) {  // Lloyd-Max levels: the products over the codes' high bits
#pragma unroll
            for (int nq = 0; nq < NQT; ++nq)
#pragma unroll
              for (int e = 0; e < 4; ++e) acch[nq][e] = 0.f;
#pragma unroll
            for (int wi = 0; wi < 2; ++wi) {
              uint32_t r0[8], r1[8];
              unpack16_hi(wi ? w0.y : w0.x, r0);
              unpack16_hi(wi ? w1.y : w1.x, r1);
#pragma unroll
              for (int k4 = 0; k4 < 4; ++k4)
#pragma unroll
                for (int nq = 0; nq < NQT; ++nq)
                  mma_f16(acch[nq], r0[2 * k4], r1[2 * k4], r0[2 * k4 + 1], r1[2 * k4 + 1], qf[4 * wi + k4][nq][0],
                          qf[4 * wi + k4][nq][1]);
            }
          }
          const uint32_t z0 = ksz[gq * C::Dg + wt], z1 = ksz[(gq + 8) * C::Dg + wt];
          const float sc0 = __half2float(__ushort_as_half(z0 & 0xffff));
          const float ze0 = __half2float(__ushort_as_half(z0 >> 16));
          const float sc1 = __half2float(__ushort_as_half(z1 & 0xffff));
          const float ze1 = __half2float(__ushort_as_half(z1 >> 16));
#pragma unroll
          for (int nq = 0; nq < NQT; ++nq) {
            if constexpr (LM) {
              const float d0 = fmaf(kLmRho, acc[nq][0] + acc[nq][1], kLmHi * (acch[nq][0] + acch[nq][1]));
              const float d1 = fmaf(kLmRho, acc[nq][2] + acc[nq][3], kLmHi * (acch[nq][2] + acch[nq][3]));
              s[0][nq][0] = fmaf(sc0, d0 * qF[nq], ze0 * qsum[nq]);
              s[0][nq][1] = fmaf(sc1, d1 * qF[nq], ze1 * qsum[nq]);
            } else {
              s[0][nq][0] = fmaf(sc0, (acc[nq][0] + acc[nq][1]) * qF[nq], ze0 * qsum[nq]);
              s[0][nq][1] = fmaf(sc1, (acc[nq][2] + acc[nq][3]) * qF[nq], ze1 * qsum[nq]);
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
            uint32_t bh0[NQT], bh1[NQT];  // Lloyd-Max levels: the high-bit pass's operands
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
              if constexpr (LM) {
                bw0[nq] = movmatrix_trans(split_f16(w0 * kLmRho));
                bw1[nq] = movmatrix_trans(split_f16(w1 * kLmRho));
                bh0[nq] = movmatrix_trans(split_f16(w0 * kLmHi));
                bh1[nq] = movmatrix_trans(split_f16(w1 * kLmHi));
              } else {
                bw0[nq] = movmatrix_trans(split_f16(w0));
                bw1[nq] = movmatrix_trans(split_f16(w1));
              }
            }
            // codes of word (wt, gq) for tokens 2cq, 2cq+1, 2cq+8, 2cq+9 of this k-step
            const int ta = 16 * ks + 2 * cq;
            const uint32_t wa = vc[(tb + ta + 0) * (C::ROWB / 4) + vcol0];
            const uint32_t wb = vc[(tb + ta + 1) * (C::ROWB / 4) + vcol1];
            const uint32_t wc = vc[(tb + ta + 8) * (C::ROWB / 4) + vcol0];
            const uint32_t wd = vc[(tb + ta + 9) * (C::ROWB / 4) + vcol1];
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              uint32_t rx[8], ry[8];
              unpack16(prmt(wa, wb, hh ? 0x7632u : 0x5410u), rx);
              unpack16(prmt(wc, wd, hh ? 0x7632u : 0x5410u), ry);
#pragma unroll
              for (int m4 = 0; m4 < 4; ++m4) {
                const int mtd = 4 * hh + m4;
#pragma unroll
                for (int nq = 0; nq < NQT; ++nq)
                  mma_f16(o[mtd][nq], rx[2 * m4], rx[2 * m4 + 1], ry[2 * m4], ry[2 * m4 + 1], bw0[nq], bw1[nq]);
              }
            }
            if constexpr (LM) {  // + kLmHi * sum of p * scale * (2 c1): the codes' high bits
#pragma unroll
              for (int hh = 0; hh < 2; ++hh) {
                uint32_t rx[8], ry[8];
                unpack16_hi(prmt(wa, wb, hh ? 0x7632u : 0x5410u), rx);
                unpack16_hi(prmt(wc, wd, hh ? 0x7632u : 0x5410u), ry);
#pragma unroll
                for (int m4 = 0; m4 < 4; ++m4) {
                  const int mtd = 4 * hh + m4;
#pragma unroll
                  for (int nq = 0; nq < NQT; ++nq)
                    mma_f16(o[mtd][nq], rx[2 * m4], rx[2 * m4 + 1], ry[2 * m4], ry[2 * m4 + 1], bh0[nq], bh1[nq]);
                }
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
          const uint32_t vb_s = smem_u32(st + (kv16 ? C::VB_V : C::BOXES * C::BOX_BYTES));
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
        ++consumed;
        if (wt == 0) issue_next();
      }
      if (o_i2) scale_o(-1);
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
      if (abort_flag) {
        aborted = true;
        break;
      }

      // ---- merge the teams of this CTA and write the segment's partial
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
        const int64_t pi = (int64_t(b) * g.Hq + head0 + hs) * a.ns + sd.slot;
        a.ws_acc[pi * D + d] = acc;
        if (d == 0) {
          a.ws_ml[pi * 2 + 0] = M;
          a.ws_ml[pi * 2 + 1] = L;
        }
      }

      // ---- the last CTA of this unit to finish merges its slots (a ticket, no
      // waiting on other CTAs), un-rotates V and stores the output
      __threadfence();
      asm volatile("bar.sync 15, %0;" ::"r"(32 * kNCW) : "memory");
      if (threadIdx.x == 0) is_last = atomicAdd(a.ticket + bh, 1) == sd.nseg - 1;
      asm volatile("bar.sync 15, %0;" ::"r"(32 * kNCW) : "memory");
      if (is_last) {
        __threadfence();
        const int nseg = sd.nseg;
        // R_V: in the CTA's last segment no copy is in flight, so at D = 128 it
        // comes into the idle stage area with one bulk copy, landing while the
        // slots are merged; otherwise its rows are read through L2
        const bool rv_smem = D == 128 && !unrot_separate(g, a.absorb_v, a.hadamard) && !a.absorb_v && !a.hadamard &&
                             !more && sg == nwin - 1 && C::NST * C::STAGE >= D * D * 4;
        const uint32_t rv_bar = smem_u32(&bars[C::NST]);
        if (rv_smem && threadIdx.x == 0) {
          mbar_arrive_expect_tx(rv_bar, D * D * 4);
          bulk_g2s(smem_u32(smem + C::OFF_STAGE), a.R_V, D * D * 4, rv_bar);
        }
        float* ob = part;                    // [G][D] merged o' (rotated basis)
        float* Ms = part + C::HEADS * D;     // [G] max, [G] sum of the merged partial
        float* Ls = Ms + C::HEADS;
        {
          // (head, 4-channel chunk) pairs f = threadIdx.x + kThreads * e.  Each
          // thread merges its head's slots online (running max, sums rescaled
          // by 2^(old max - new max); every thread of a head takes the same
          // steps), in groups of SU slots whose loads are all issued before
          // any is used: a unit shared by many CTAs costs a few L2 round trips
          constexpr int D4 = D / 4;
          constexpr int IPT4 = C::HEADS * D4 / kThreads;
          constexpr int SU = IPT4 >= 8 ? 1 : 16 / IPT4;
          static_assert(IPT4 * kThreads == C::HEADS * D4, "whole float4 chunks per thread");
          float4 acc[IPT4];
          float Mr[IPT4], Lr[IPT4];
#pragma unroll
          for (int e = 0; e < IPT4; ++e) {
            acc[e] = make_float4(0.f, 0.f, 0.f, 0.f);
            Mr[e] = -INFINITY;
            Lr[e] = 0.f;
          }
          for (int sp0 = 0; sp0 < nseg; sp0 += SU) {
            float4 v[SU][IPT4];
            float2 ml[SU][IPT4];
#pragma unroll
            for (int j = 0; j < SU; ++j)
#pragma unroll
              for (int e = 0; e < IPT4; ++e) {
                const int f = threadIdx.x + kThreads * e, i = f / D4, d4 = f % D4;
                v[j][e] = make_float4(0.f, 0.f, 0.f, 0.f);
                ml[j][e] = make_float2(-INFINITY, 0.f);
                if (i < Gh && sp0 + j < nseg) {
                  const int64_t si = (int64_t(b) * g.Hq + head0 + i) * a.ns + sp0 + j;
                  v[j][e] = __ldcg(reinterpret_cast<const float4*>(a.ws_acc + si * D) + d4);
                  ml[j][e] = __ldcg(reinterpret_cast<const float2*>(a.ws_ml) + si);
                }
              }
            // one rescale per group to the group's max, then independent
            // weights (an empty partial or a missing slot carries (-inf, 0)
            // and a zero vector, so its weight is 0)
#pragma unroll
            for (int e = 0; e < IPT4; ++e) {
              float mg = Mr[e];
#pragma unroll
              for (int j = 0; j < SU; ++j) mg = fmaxf(mg, ml[j][e].x);
              if (mg != -INFINITY) {
                const float co = ex2(Mr[e] - mg);
                acc[e].x *= co;
                acc[e].y *= co;
                acc[e].z *= co;
                acc[e].w *= co;
                Lr[e] *= co;
#pragma unroll
                for (int j = 0; j < SU; ++j) {
                  const float cn = ex2(ml[j][e].x - mg);
                  acc[e].x = fmaf(v[j][e].x, cn, acc[e].x);
                  acc[e].y = fmaf(v[j][e].y, cn, acc[e].y);
                  acc[e].z = fmaf(v[j][e].z, cn, acc[e].z);
                  acc[e].w = fmaf(v[j][e].w, cn, acc[e].w);
                  Lr[e] = fmaf(ml[j][e].y, cn, Lr[e]);
                }
                Mr[e] = mg;
              }
            }
          }
#pragma unroll
          for (int e = 0; e < IPT4; ++e) {
            const int f = threadIdx.x + kThreads * e, i = f / D4;
            if (i < Gh) {
              const float inv = Lr[e] > 0.f ? 1.f / Lr[e] : 0.f;
              reinterpret_cast<float4*>(ob)[f] =
                  make_float4(acc[e].x * inv, acc[e].y * inv, acc[e].z * inv, acc[e].w * inv);
              if (f % D4 == 0) {
                Ms[i] = Mr[e];
                Ls[i] = Lr[e];
              }
            }
          }
        }
        asm volatile("bar.sync 15, %0;" ::"r"(32 * kNCW) : "memory");
        bool rv_ok = true;
        if (rv_smem) {
          rv_ok = mbar_wait(rv_bar, 0, a.wait_ns);
          if (!rv_ok && threadIdx.x == 0) status_or(a.status, OSCAR_DEV_TIMEOUT);
        }
        auto store = [&](int i, int r, float v) {
          const int64_t oi = (int64_t(b) * g.Hq + head0 + i) * D + r;
          if (a.out_fp32)
            static_cast<float*>(a.out)[oi] = v;
          else
            static_cast<__nv_bfloat16*>(a.out)[oi] = __float2bfloat16_rn(v);
        };
        if (a.hadamard && !a.absorb_v) {
          // o = o' H (the in-quant Hadamard is symmetric): warp w transforms
          // the (head, group) pairs w, w + kNCW, ... in registers
          for (int pr = warp; pr < Gh * C::Dg; pr += kNCW) {
            const int i = pr / C::Dg, j = pr % C::Dg;
            float x[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) x[e] = ob[i * D + j * kGroup + lane + 32 * e];
            hadamard128_warp(x, lane);
#pragma unroll
            for (int e = 0; e < 4; ++e) store(i, j * kGroup + lane + 32 * e, x[e]);
          }
        } else if (!unrot_separate(g, a.absorb_v, a.hadamard)) {
          // o = o' R_V^T (or o' when absorbed): one thread per output channel r.
          // At head_dim 128, R_V comes from the stage area when it was
          // prefetched there, else from L2, through the same arithmetic in the
          // same order, so the output does not depend on which CTA merges.
          const float* rvs = (rv_smem && rv_ok) ? reinterpret_cast<const float*>(smem + C::OFF_STAGE) : nullptr;
          for (int r = threadIdx.x; r < D; r += 32 * kNCW) {
            float res[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) res[i] = 0.f;
            if (a.absorb_v) {
#pragma unroll
              for (int i = 0; i < 8; ++i)
                if (i < Gh) res[i] = ob[i * D + r];
            } else {
              // 16-byte loads in a skewed walk over j: thread r reads chunk
              // (j4 + r) % (D / 4) of row r and of each o' row, so the eight
              // threads of a quarter warp touch eight different chunks
              const float4* rv4 = reinterpret_cast<const float4*>(rvs ? rvs + r * D : a.R_V + int64_t(r) * D);
#pragma unroll 4
              for (int j4 = 0; j4 < D / 4; ++j4) {
                const int jq = (j4 + r) & (D / 4 - 1);
                const float4 rv = rvs ? rv4[jq] : __ldg(rv4 + jq);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                  if (i < Gh) {
                    const float4 ov = *reinterpret_cast<const float4*>(ob + i * D + 4 * jq);
                    res[i] = fmaf(rv.x, ov.x, fmaf(rv.y, ov.y, fmaf(rv.z, ov.z, fmaf(rv.w, ov.w, res[i]))));
                  }
                }
              }
            }
#pragma unroll
            for (int i = 0; i < 8; ++i)
              if (i < Gh) store(i, r, res[i]);
          }
        } else {
          // o' goes to the unit's workspace slot 0 (every slot has been read)
          // and unrot_kernel applies R_V^T for all units at once, spread over
          // the GPU (see unrot_separate)
          for (int e = threadIdx.x; e < Gh * (D / 4); e += kThreads) {
            const int i = e / (D / 4), j4 = e % (D / 4);
            const int64_t si = (int64_t(b) * g.Hq + head0 + i) * a.ns;
            __stcg(reinterpret_cast<float4*>(a.ws_acc + si * D) + j4, reinterpret_cast<const float4*>(ob + i * D)[j4]);
          }
        }
        if (threadIdx.x < Gh && a.lse) {
          const int i = threadIdx.x;
          const float M = Ms[i], L = Ls[i];
          a.lse[int64_t(b) * g.Hq + head0 + i] =
              (M == -INFINITY || !(L > 0.f)) ? -INFINITY : (M + log2f(L)) * 0.6931471805599453f;
        }
      }
      // part and the shared q' fragments are rewritten by the next segment
      asm volatile("bar.sync 15, %0;" ::"r"(32 * kNCW) : "memory");
      if (sg + 1 < nwin) qb_issue(seg[sg + 1].b, seg[sg + 1].h);
    }  // segments
    if (aborted || !more) break;
    __syncthreads();  // the table is rebuilt for the next window
  }  // windows

  // after an early exit, wait (bounded) for copies still landing in our stages
  // and in the shared q' image
  // (each wait is bounded and none is skipped: a stage whose barrier never
  // completes does not stop the wait for the copies of the later ones)
  if (wt == 0 && lane == 0)
    for (int jj = consumed; jj < issued; ++jj) (void)mbar_wait(smem_u32(&bars[my_stage(jj)]), (jj / C::NSTW) & 1, a.wait_ns);
  if (threadIdx.x == 0)
    for (; qb_waited < qb_issued; ++qb_waited) (void)mbar_wait(qb_bar, qb_waited & 1, a.wait_ns);
}

// ---------------------------------------------------------------------------
// host launch
// ---------------------------------------------------------------------------
// ---------------------------------------------------------------------------
// o = o' R_V^T at head_dim 256 / 512 (V not absorbed, no in-quant Hadamard):
// the split kernel leaves the merged o' of every (sequence, query head) in its
// workspace slot 0.  CTA (x, y) holds rows [16 x, 16 x + 16) of R_V in shared
// memory; each warp takes one (sequence, head) vector at a time, lane l
// multiplies its float4 chunks l, l + 32, ... of o' with the 16 rows, and a
// halving butterfly leaves the sum of output r0 + (l >> 1) in lanes l.
// Empty sequences keep the output qrot wrote.
// ---------------------------------------------------------------------------
constexpr int kUnrotRows = 16;
// unrot_kernel runs after the split kernel (the decode's fourth launch)
inline bool unrot_launched(const DecodeArgs& a) { return unrot_separate(a.g, a.absorb_v, a.hadamard); }
constexpr int kUnrotThreads = 256;

template <int W, int SH>
__device__ __forceinline__ void butterfly_half(float (&res)[kUnrotRows], int lane) {
  const bool up = (lane & SH) != 0;
#pragma unroll
  for (int i = 0; i < W; ++i) {
    const float send = up ? res[i] : res[i + W];
    const float recv = __shfl_xor_sync(0xffffffffu, send, SH);
    res[i] = (up ? res[i + W] : res[i]) + recv;
  }
}

template <int D>
__global__ void __launch_bounds__(kUnrotThreads, 1) unrot_kernel(const DecodeArgs a) {
  __shared__ __align__(16) float rv[kUnrotRows][D];
  __shared__ __align__(8) uint64_t rv_bar;
  __shared__ int rv_ok;
  const int r0 = blockIdx.x * kUnrotRows;
  // R_V's rows arrive with one bulk copy, issued before the wait for the split
  // kernel (they do not depend on it)
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&rv_bar), 1);
    mbar_fence_init();
    mbar_arrive_expect_tx(smem_u32(&rv_bar), kUnrotRows * D * 4);
    bulk_g2s(smem_u32(&rv[0][0]), a.R_V + int64_t(r0) * D, kUnrotRows * D * 4, smem_u32(&rv_bar));
  }
  pdl_wait();  // the split kernel's merges are complete
  if (threadIdx.x == 0) {
    rv_ok = mbar_wait(smem_u32(&rv_bar), 0, a.wait_ns);
    if (!rv_ok) status_or(a.status, OSCAR_DEV_TIMEOUT);
  }
  __syncthreads();
  if (!rv_ok) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nvec = a.g.B * a.g.Hq;
  constexpr int C4 = D / 128;  // float4 chunks of o' per lane
  for (int vi = blockIdx.y * (kUnrotThreads / 32) + warp; vi < nvec; vi += gridDim.y * (kUnrotThreads / 32)) {
    if (clamp_seq_len(a, vi / a.g.Hq) == 0) continue;
    const float4* op = reinterpret_cast<const float4*>(a.ws_acc + int64_t(vi) * a.ns * D);
    float4 o[C4];
#pragma unroll
    for (int k = 0; k < C4; ++k) o[k] = __ldcg(op + lane + 32 * k);
    float res[kUnrotRows];
#pragma unroll
    for (int rr = 0; rr < kUnrotRows; ++rr) {
      float acc = 0.f;
#pragma unroll
      for (int k = 0; k < C4; ++k) {
        const float4 r4 = reinterpret_cast<const float4*>(&rv[rr][0])[lane + 32 * k];
        acc = fmaf(r4.x, o[k].x, fmaf(r4.y, o[k].y, fmaf(r4.z, o[k].z, fmaf(r4.w, o[k].w, acc))));
      }
      res[rr] = acc;
    }
    // halving butterfly: after the step over lane bit s, a lane keeps the half
    // of its values that its bit s selects, summed with its partner's
    butterfly_half<8, 16>(res, lane);
    butterfly_half<4, 8>(res, lane);
    butterfly_half<2, 4>(res, lane);
    butterfly_half<1, 2>(res, lane);
    res[0] += __shfl_xor_sync(0xffffffffu, res[0], 1);
    if ((lane & 1) == 0) {
      const int64_t oi = int64_t(vi) * D + r0 + (lane >> 1);
      if (a.out_fp32)
        static_cast<float*>(a.out)[oi] = res[0];
      else
        static_cast<__nv_bfloat16*>(a.out)[oi] = __float2bfloat16_rn(res[0]);
    }
  }
}

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
  int occ[3][2][2][2] = {};  // [head_dim][G > 4][V kept BF16][Lloyd-Max levels]
  bool ready = false;
};
DevInfo g_dev[64];

template <int D, int NQT, bool VB, bool LM>
int prepare_split(int dev) {
  using C = DecCfg<D, NQT>;
  if (cudaFuncSetAttribute(split_kernel<D, NQT, VB, LM>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) !=
      cudaSuccess)
    return -1;
  int occ = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, split_kernel<D, NQT, VB, LM>, kThreads, C::SMEM) !=
      cudaSuccess)
    return -1;
  return occ;
}

int didx(int D) { return D == 128 ? 0 : (D == 256 ? 1 : 2); }

template <int D>
bool prepare_d(int dev, DevInfo& di) {
  const int o[8] = {prepare_split<D, 1, false, false>(dev), prepare_split<D, 1, true, false>(dev),
                    prepare_split<D, 2, false, false>(dev), prepare_split<D, 2, true, false>(dev),
                    prepare_split<D, 1, false, true>(dev),  prepare_split<D, 1, true, true>(dev),
                    prepare_split<D, 2, false, true>(dev),  prepare_split<D, 2, true, true>(dev)};
  for (int k = 0; k < 8; ++k) {
    if (o[k] <= 0) return false;
    di.occ[didx(D)][(k / 2) % 2][k % 2][k / 4] = o[k];
  }
  return true;
}

int dinfo_init(int dev) {
  DevInfo& di = g_dev[dev];
  if (di.ready) return 0;
  if (cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
  if (!prepare_d<128>(dev, di) || !prepare_d<256>(dev, di) || !prepare_d<512>(dev, di)) return -1;
  di.ready = true;
  return 0;
}

template <int D, int NQT, bool VB, bool LM>
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
  if (g.S > 0 && !encode_rows_bf16(&maps[0], kb, bh * g.S, D, 64, kBfTok)) return OSCAR_ERR_LAUNCH;
  if (g.W > 0 && !encode_rows_bf16(&maps[2], kb + g.sink_bytes, bh * g.W, D, 64, kBfTok)) return OSCAR_ERR_LAUNCH;
  if (g.vb) {
    // V kept BF16: one map over its [B*Hkv*cap][D] rows, indexed by position
    if (!encode_rows_bf16(&maps[1], vb, bh * uint64_t(g.cap), D, 64, kBfTok)) return OSCAR_ERR_LAUNCH;
  } else {
    if (g.S > 0 && !encode_rows_bf16(&maps[1], vb, bh * g.S, D, 64, kBfTok)) return OSCAR_ERR_LAUNCH;
    if (g.W > 0 && !encode_rows_bf16(&maps[3], vb + g.sink_bytes, bh * g.W, D, 64, kBfTok)) return OSCAR_ERR_LAUNCH;
  }
  // INT2 code rows [B*Hkv*ncap][D/4] per role, 128-row swizzled boxes (unused with V kept BF16)
  CUtensorMap cmaps[2];
  std::memset(cmaps, 0, sizeof(cmaps));
  const uint64_t crows = bh * uint64_t(g.ncap);
  if (C::SWZ && !g.vb && crows > 0) {
    if (crows >= (uint64_t(1) << 31)) return OSCAR_ERR_LAUNCH;  // 32-bit TMA row coordinates
    const uint64_t codes_off = g.sink_bytes + g.ring_bytes;
    if (!encode_code_rows(&cmaps[0], kb + codes_off, crows, C::ROWB, kI2Tok) ||
        !encode_code_rows(&cmaps[1], vb + codes_off, crows, C::ROWB, kI2Tok))
      return OSCAR_ERR_LAUNCH;
  }
  if (launch_pdl(split_kernel<D, NQT, VB, LM>, dim3(unsigned(a.ctas)), dim3(kThreads), C::SMEM, stream, maps[0], maps[1],
                 maps[2], maps[3], cmaps[0], cmaps[1], a) != cudaSuccess)
    return OSCAR_ERR_LAUNCH;
  if (unrot_launched(a)) {
    const int nvec = g.B * g.Hq, wpc = kUnrotThreads / 32;
    const int gy = std::max(1, std::min((nvec + wpc - 1) / wpc, 8));
    if (launch_pdl(unrot_kernel<D>, dim3(D / kUnrotRows, unsigned(gy)), dim3(kUnrotThreads), 0, stream, a) !=
        cudaSuccess)
      return OSCAR_ERR_LAUNCH;
  }
  if (prof && cudaEventRecord(g_prof_stop, stream) != cudaSuccess) return OSCAR_ERR_LAUNCH;
  return OSCAR_OK;
}

}  // namespace

thread_local cudaEvent_t g_prof_start = nullptr, g_prof_stop = nullptr;
thread_local uint64_t g_test_wait_ns = 0;
thread_local int g_test_wait_poison = 0;

int decode_kernel_count(const Geom& g, bool absorb_v, bool hadamard) {
  return 2 + (unrot_separate(g, absorb_v, hadamard) ? 1 : 0);
}

uint64_t decode_workspace_bytes(const Geom& g, int ns) {
  const uint64_t bq = uint64_t(g.B) * g.Hq, units = uint64_t(g.B) * g.Hkv;
  const uint64_t nqt = g.G > 4 ? 2 : 1;
  return align256(units * g.Dg * nqt * 2048) + align256(units * g.Dg * nqt * 4096) + align256(bq * g.Dg * 4) +
         align256(bq * g.Dg * 4) + align256(bq * ns * g.D * 4) + align256(bq * ns * 2 * 4) + align256(units * 4);
}

int decode_grid(const Geom& g, int seq_len_hint, int num_splits) {
  const int64_t units = int64_t(g.B) * g.Hkv;
  if (num_splits > 0) return int(std::min<int64_t>(int64_t(num_splits) * units, 1 << 30));
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev >= 64 || dinfo_init(dev) != 0) return -1;
  const DevInfo& di = g_dev[dev];
  // persistent: as many CTAs as are resident at once; for short contexts
  // fewer, so that each team still gets about one block of the cache a
  // context of seq_len_hint implies (a CTA's fixed cost, ~10 us of set-up and
  // merge, runs in parallel with the others, so small problems spread wide)
  const int64_t resident = int64_t(di.sms) * di.occ[didx(g.D)][g.G > 4 ? 1 : 0][g.vb ? 1 : 0][g.lm ? 1 : 0];
  const Regions r = make_regions(seq_len_hint, g.S, g.W, g.D, g.vb, g.lm);
  const int64_t min_cost = int64_t(kNCW / g.Dg) * r.cbf;
  const int64_t by_work = std::max<int64_t>(1, unit_cost(r) * units / min_cost);
  return int(std::max<int64_t>(1, std::min(resident, by_work)));
}

template <bool VB, bool LM>
int launch_decode_mode(const DecodeArgs& a, cudaStream_t stream) {
  const bool big = a.g.G > 4;
  switch (a.g.D) {
    case 128: return big ? launch_decode_d<128, 2, VB, LM>(a, stream) : launch_decode_d<128, 1, VB, LM>(a, stream);
    case 256: return big ? launch_decode_d<256, 2, VB, LM>(a, stream) : launch_decode_d<256, 1, VB, LM>(a, stream);
    case 512: return big ? launch_decode_d<512, 2, VB, LM>(a, stream) : launch_decode_d<512, 1, VB, LM>(a, stream);
    default: return OSCAR_ERR_UNSUPPORTED;
  }
}

int launch_decode(const DecodeArgs& a, cudaStream_t stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev >= 64 || dinfo_init(dev) != 0) return OSCAR_ERR_LAUNCH;
  if (a.g.vb) return a.g.lm ? launch_decode_mode<true, true>(a, stream) : launch_decode_mode<true, false>(a, stream);
  return a.g.lm ? launch_decode_mode<false, true>(a, stream) : launch_decode_mode<false, false>(a, stream);
}

}  // namespace oscar
