// Calibration of the rotations from activations:
//   K side: Sigma = Q^T Q in float64, its eigenvectors by one-sided Jacobi in
//   float64, sorted by descending eigenvalue with a sign convention, then
//   R_K = E H_D P_br;
//   V side: the same from Sigma_V = sum_t w_t v_t^T v_t, each key/value row
//   weighted by its score energy w_t = k_t Q^T Q k_t^T (the sum over the
//   calibration queries of the squared logit q . k_t).
//
// Source: "OSCAR-RotationZoo" model card (File format: R_K = R H P_br with R
// the eigenvectors of the query covariance, H a head-dim Hadamard and P_br the
// eigenvalue-sorted bit-reversal permutation; for V, the covariance of the
// value rows weighted by attention scores, printed as V^T diag(K^T (Q^T Q) K) V
// and read with K holding the keys as columns) and the hysenlabs article on OSCAR (How the offline
// rotation is fit: Q/K/V activations are captured offline and the rotation is
// derived from their covariance).
//
// Offline work, not on the decode path.  Kernels on the caller's stream:
//   cov_kernel       Sigma += X^T diag(w) X: CTA (i, j, c) accumulates the
//                    64 x 64 tile (i, j) of Sigma over row chunk c in float64
//                    (a product of two float32 values is exact in float64; a
//                    row weight adds one rounding; each thread a 4 x 4 register
//                    block) and adds it into Sigma with float64 atomics;
//   weight_kernel    (V side) w_t = k_t Sigma_Q k_t^T: thread j of a CTA of D
//                    threads forms column j of k Sigma_Q for 16 key rows, the
//                    CTA reduces each row's dot product with k;
//   jacobi_kernel    cooperative grid, one CTA per column pair: one-sided
//                    Jacobi on Sigma (below);
//   finalize_kernel  one CTA, one thread per eigenpair / row: rank the
//                    eigenvalues, move each eigenvector to its rank, sign it,
//                    apply H_D to every row with float64 butterflies and write
//                    column j of the result from column br(j), as float32.
#include <cooperative_groups.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "internal.h"

namespace oscar {
namespace {

constexpr int kCovTile = 64;          // Sigma tile per CTA
constexpr int kCovRows = 32;          // rows staged per step
constexpr int64_t kCovChunk = 4096;   // rows per CTA
// the row chunks are the grid's z dimension (at most 65535)
static_assert(OSCAR_KV_CALIB_MAX_ROWS == 65535 * kCovChunk, "calibration row limit");
constexpr int kMaxSweeps = 40;
constexpr int kPairThreads = 256;

// Sigma tile (ti, tj) += X^T diag(w) X over one chunk of rows (w NULL: all
// weights 1); thread (ty, tx) owns a 4 x 4 block of the 64 x 64 tile; rows are
// staged as float64 (exact), the first operand times its row's weight.
__global__ void __launch_bounds__(256) cov_kernel(const float* __restrict__ q, int64_t n, int D,
                                                  const double* __restrict__ wrow, double* __restrict__ sigma) {
  __shared__ double sa[kCovRows][kCovTile], sb[kCovRows][kCovTile];
  const int ti = blockIdx.x, tj = blockIdx.y;
  const int t = threadIdx.x, ty = t >> 4, tx = t & 15;
  const int64_t row_lo = int64_t(blockIdx.z) * kCovChunk;
  const int64_t row_hi = row_lo + kCovChunk < n ? row_lo + kCovChunk : n;
  double acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.0;
  for (int64_t row0 = row_lo; row0 < row_hi; row0 += kCovRows) {
    for (int idx = t; idx < kCovRows * kCovTile; idx += 256) {
      const int rr = idx / kCovTile, cc = idx % kCovTile;
      const int64_t row = row0 + rr;
      const bool in = row < row_hi;
      sa[rr][cc] = in ? double(q[row * D + ti * kCovTile + cc]) * (wrow ? wrow[row] : 1.0) : 0.0;
      sb[rr][cc] = in ? double(q[row * D + tj * kCovTile + cc]) : 0.0;
    }
    __syncthreads();
#pragma unroll 4
    for (int rr = 0; rr < kCovRows; ++rr) {
      double a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        a[i] = sa[rr][ty * 4 + i];
        b[i] = sb[rr][tx * 4 + i];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fma(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j)
      atomicAdd(&sigma[int64_t(ti * kCovTile + ty * 4 + i) * D + tj * kCovTile + tx * 4 + j], acc[i][j]);
}

constexpr int kWTok = 16;  // key rows per weight_kernel CTA

// w[t] = k_t Sigma_Q k_t^T for kWTok key rows; blockDim.x == D (Sigma_Q is
// symmetric, so thread j reads column j as row j's transpose: coalesced).
__global__ void __launch_bounds__(512) weight_kernel(const float* __restrict__ k, int64_t n, int D,
                                                     const double* __restrict__ sq, double* __restrict__ w) {
  __shared__ float ks[kWTok][512];
  __shared__ double red[kWTok][16];
  const int j = threadIdx.x;
  const int64_t t0 = int64_t(blockIdx.x) * kWTok;
  for (int r = 0; r < kWTok; ++r) ks[r][j] = t0 + r < n ? k[(t0 + r) * D + j] : 0.f;
  __syncthreads();
  double y[kWTok];
#pragma unroll
  for (int r = 0; r < kWTok; ++r) y[r] = 0.0;
  for (int i = 0; i < D; ++i) {
    const double sij = sq[int64_t(i) * D + j];
#pragma unroll
    for (int r = 0; r < kWTok; ++r) y[r] = fma(double(ks[r][i]), sij, y[r]);
  }
  const int warp = j >> 5, lane = j & 31, nw = D >> 5;
#pragma unroll
  for (int r = 0; r < kWTok; ++r) {
    double v = y[r] * double(ks[r][j]);
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0) red[r][warp] = v;
  }
  __syncthreads();
  if (j < kWTok && t0 + j < n) {
    double tot = 0.0;
    for (int q = 0; q < nw; ++q) tot += red[j][q];
    w[t0 + j] = tot;
  }
}

// Sum of v over the block (every thread gets it); red has blockDim / 32 slots.
__device__ double block_sum(double v, double* red) {
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[w] = v;
  __syncthreads();
  double s = 0.0;
  for (int i = 0; i < nw; ++i) s += red[i];
  return s;
}

// One-sided (Hestenes) Jacobi on Sigma: columns of A (= Sigma, stored by
// columns; Sigma is symmetric) are rotated in pairs until mutually
// orthogonal, V accumulates the rotations.  For a symmetric positive
// semi-definite Sigma the result is its eigendecomposition: A = Sigma V with
// column norms equal to the eigenvalues.  Round r pairs the columns by the
// circle method (column D-1 fixed); its D/2 pairs are independent, so the
// CTAs of one cooperative grid take whole pairs (three block-reduced dot
// products, then the two columns of A and of V) and meet at one grid barrier
// per round.  A sweep (D-1 rounds) ends with the largest |cos| between the
// pairs it rotated; below 1e-15 the grid stops, at kMaxSweeps sweeps it stops
// and flags OSCAR_DEV_NOT_CONVERGED.  Every loop is bounded.
__global__ void __launch_bounds__(kPairThreads) jacobi_kernel(double* __restrict__ A, double* __restrict__ V,
                                                              int D, unsigned long long* __restrict__ sweep_max,
                                                              int32_t* status, int32_t* info) {
  namespace cg = cooperative_groups;
  cg::grid_group grid = cg::this_grid();
  __shared__ double red[kPairThreads / 32];
  const int tid = threadIdx.x, nt = blockDim.x;
  const int64_t DD = int64_t(D) * D;
  for (int64_t idx = int64_t(blockIdx.x) * nt + tid; idx < DD; idx += int64_t(gridDim.x) * nt)
    V[idx] = (idx / D == idx % D) ? 1.0 : 0.0;
  if (blockIdx.x == 0 && tid < 2) sweep_max[tid] = 0ull;
  grid.sync();
  const int half = D / 2;
  int sweep = 0;
  bool converged = false;
  for (; sweep < kMaxSweeps; ++sweep) {
    double worst = 0.0;  // largest |cos| this CTA saw (uniform across the CTA)
    for (int rnd = 0; rnd < D - 1; ++rnd) {
      for (int k = blockIdx.x; k < half; k += gridDim.x) {
        int p = k == 0 ? rnd : (rnd + k) % (D - 1);
        int q = k == 0 ? D - 1 : (rnd - k + (D - 1)) % (D - 1);
        if (p > q) {
          const int x = p;
          p = q;
          q = x;
        }
        double* ap = A + int64_t(p) * D;
        double* aq = A + int64_t(q) * D;
        double al = 0.0, be = 0.0, ga = 0.0;
        for (int i = tid; i < D; i += nt) {
          const double x = ap[i], y = aq[i];
          al += x * x;
          be += y * y;
          ga += x * y;
        }
        al = block_sum(al, red);
        be = block_sum(be, red);
        ga = block_sum(ga, red);
        const double nrm = sqrt(al * be);
        if (!isfinite(al) || !isfinite(be) || !isfinite(ga)) {
          // a non-finite covariance (non-finite calibration rows): flag it and
          // let the sweep count run out instead of reporting convergence
          if (tid == 0) status_or(status, OSCAR_DEV_NONFINITE);
          worst = INFINITY;
        } else if (ga != 0.0 && nrm > 0.0) {
          worst = fmax(worst, fabs(ga) / nrm);
          const double zeta = (be - al) / (2.0 * ga);
          const double az = fabs(zeta);
          const double tt = az > 1e150 ? 0.5 / az : 1.0 / (az + sqrt(1.0 + zeta * zeta));
          const double tv = zeta < 0.0 ? -tt : tt;
          const double c = 1.0 / sqrt(1.0 + tv * tv), s = c * tv;
          double* vp = V + int64_t(p) * D;
          double* vq = V + int64_t(q) * D;
          for (int i = tid; i < D; i += nt) {
            const double x = ap[i], y = aq[i];
            ap[i] = c * x - s * y;
            aq[i] = s * x + c * y;
            const double u = vp[i], w = vq[i];
            vp[i] = c * u - s * w;
            vq[i] = s * u + c * w;
          }
        }
        __syncthreads();
      }
      grid.sync();
    }
    // largest |cos| of the sweep over the grid (non-negative doubles order as integers)
    if (tid == 0) atomicMax(&sweep_max[sweep & 1], static_cast<unsigned long long>(__double_as_longlong(worst)));
    grid.sync();
    const double m = __longlong_as_double(static_cast<long long>(sweep_max[sweep & 1]));
    if (blockIdx.x == 0 && tid == 0) sweep_max[(sweep + 1) & 1] = 0ull;
    grid.sync();
    if (m <= 1e-15) {
      converged = true;
      ++sweep;
      break;
    }
  }
  if (blockIdx.x == 0 && tid == 0) {
    info[0] = sweep;
    if (!converged) status_or(status, OSCAR_DEV_NOT_CONVERGED);
  }
}

// One CTA, thread i per eigenpair / column / row: eigenvalue i = |column i of
// A| (A = Sigma V), rank by descending eigenvalue (ties by index), move column
// i of V to column rank of E, sign it (largest-magnitude entry, the first on
// ties, positive), then each row of E times H_D (in-place butterflies, 1/sqrt D)
// and column j of R from column br(j).
__global__ void finalize_kernel(const double* __restrict__ A, const double* __restrict__ V,
                                double* __restrict__ lam, double* __restrict__ E, float* __restrict__ R, int D,
                                int32_t* status) {
  const int i = threadIdx.x;
  double n2 = 0.0;
  for (int r = 0; r < D; ++r) {
    const double a = A[int64_t(i) * D + r];
    n2 += a * a;
  }
  // a non-finite eigenvalue is flagged and ranks last (as -inf), so the ranks
  // stay a permutation (ties by index) and every column of E is written
  const double l0 = sqrt(n2);
  if (!isfinite(l0)) status_or(status, OSCAR_DEV_NONFINITE);
  lam[i] = isfinite(l0) ? l0 : -INFINITY;
  __syncthreads();
  const double li = lam[i];
  int rank = 0;
  for (int j = 0; j < D; ++j) {
    const double lj = lam[j];
    rank += (lj > li || (lj == li && j < i)) ? 1 : 0;
  }
  for (int r = 0; r < D; ++r) E[int64_t(r) * D + rank] = V[int64_t(i) * D + r];
  __syncthreads();
  int piv = 0;
  double best = -1.0;
  for (int r = 0; r < D; ++r) {
    const double a = fabs(E[int64_t(r) * D + i]);
    if (a > best) {
      best = a;
      piv = r;
    }
  }
  if (E[int64_t(piv) * D + i] < 0.0)
    for (int r = 0; r < D; ++r) E[int64_t(r) * D + i] = -E[int64_t(r) * D + i];
  __syncthreads();
  double* x = E + int64_t(i) * D;
  for (int len = 1; len < D; len <<= 1)
    for (int k = 0; k < D; k += 2 * len)
      for (int m = k; m < k + len; ++m) {
        const double a = x[m], b = x[m + len];
        x[m] = a + b;
        x[m + len] = a - b;
      }
  const double inv = 1.0 / sqrt(double(D));
  const int bits = __ffs(D) - 1;
  for (int j = 0; j < D; ++j) {
    const int src = int(__brev(unsigned(j)) >> (32 - bits));
    R[int64_t(i) * D + j] = float(x[src] * inv);
  }
}

// Workspace: A (Sigma, then Sigma V by columns), V, E (on the V side first
// Sigma_Q), the eigenvalues, the sweep maxima and info; then (V side) the row
// weights.
struct CalibWs {
  double *A, *V, *E, *lam;
  unsigned long long* sweep_max;
  int32_t* info;
  double* w;
};

CalibWs calib_ws(void* ws, int D) {
  uint8_t* b = static_cast<uint8_t*>(ws);
  const uint64_t mat = align256(uint64_t(D) * D * 8);
  CalibWs c;
  c.A = reinterpret_cast<double*>(b);
  c.V = reinterpret_cast<double*>(b + mat);
  c.E = reinterpret_cast<double*>(b + 2 * mat);
  c.lam = reinterpret_cast<double*>(b + 3 * mat);
  c.sweep_max = reinterpret_cast<unsigned long long*>(b + 3 * mat + align256(uint64_t(D) * 8));
  c.info = reinterpret_cast<int32_t*>(c.sweep_max + 2);
  c.w = reinterpret_cast<double*>(b + calibrate_workspace_bytes(D));
  return c;
}

// Sigma (zeroed here) += X^T diag(w) X over the n rows of x
int launch_cov(const float* x, int64_t n, int D, const double* w, double* sigma, cudaStream_t stream) {
  if (cudaMemsetAsync(sigma, 0, size_t(D) * D * 8, stream) != cudaSuccess) return OSCAR_ERR_LAUNCH;
  const int64_t chunks = (n + kCovChunk - 1) / kCovChunk;
  cov_kernel<<<dim3(D / kCovTile, D / kCovTile, unsigned(chunks)), 256, 0, stream>>>(x, n, D, w, sigma);
  return cudaGetLastError() == cudaSuccess ? OSCAR_OK : OSCAR_ERR_LAUNCH;
}

// R = E H_D P_br from the covariance in c.A (overwritten)
int launch_fit(CalibWs& c, int D, float* R, int32_t* status, cudaStream_t stream) {
  double* A = c.A;
  double* V = c.V;
  unsigned long long* sweep_max = c.sweep_max;
  int32_t* info = c.info;
  // one CTA per column pair, as many as can be resident together
  int dev = 0, sms = 0, per_sm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, jacobi_kernel, kPairThreads, 0) != cudaSuccess || per_sm < 1)
    return OSCAR_ERR_LAUNCH;
  const int grid = std::min(D / 2, sms * per_sm);
  void* args[] = {&A, &V, &D, &sweep_max, &status, &info};
  if (cudaLaunchCooperativeKernel(reinterpret_cast<void*>(jacobi_kernel), dim3(grid), dim3(kPairThreads), args, 0,
                                  stream) != cudaSuccess)
    return OSCAR_ERR_LAUNCH;
  finalize_kernel<<<1, D, 0, stream>>>(A, V, c.lam, c.E, R, D, status);
  return cudaGetLastError() == cudaSuccess ? OSCAR_OK : OSCAR_ERR_LAUNCH;
}

}  // namespace

uint64_t calibrate_workspace_bytes(int D) { return 3 * align256(uint64_t(D) * D * 8) + align256(uint64_t(D) * 8) + 256; }

uint64_t calibrate_rv_workspace_bytes(int D, int64_t n_kv) {
  return calibrate_workspace_bytes(D) + align256(uint64_t(n_kv) * 8);
}

int launch_calibrate(const float* q, int64_t n, int D, float* R, void* ws, int32_t* status, cudaStream_t stream) {
  CalibWs c = calib_ws(ws, D);
  const int rc = launch_cov(q, n, D, nullptr, c.A, stream);
  if (rc != OSCAR_OK) return rc;
  return launch_fit(c, D, R, status, stream);
}

int launch_calibrate_rv(const float* q, int64_t nq, const float* k, const float* v, int64_t nkv, int D, float* R,
                        void* ws, int32_t* status, cudaStream_t stream) {
  CalibWs c = calib_ws(ws, D);
  int rc = launch_cov(q, nq, D, nullptr, c.E, stream);  // Sigma_Q (E is free until the fit's last kernel)
  if (rc != OSCAR_OK) return rc;
  weight_kernel<<<unsigned((nkv + kWTok - 1) / kWTok), D, 0, stream>>>(k, nkv, D, c.E, c.w);
  if (cudaGetLastError() != cudaSuccess) return OSCAR_ERR_LAUNCH;
  rc = launch_cov(v, nkv, D, c.w, c.A, stream);
  if (rc != OSCAR_OK) return rc;
  return launch_fit(c, D, R, status, stream);
}

}  // namespace oscar
