// Calibration of the K-side rotation from query activations:
// Sigma = Q^T Q in float64, its eigenvectors by one-sided Jacobi in float64,
// sorted by descending eigenvalue with a sign convention, then
// R_K = E H_D P_br.
//
// Source: "OSCAR-RotationZoo" model card (File format: R_K = R H P_br with R
// the eigenvectors of the query covariance, H a head-dim Hadamard and P_br the
// eigenvalue-sorted bit-reversal permutation) and the hysenlabs article on
// OSCAR (How the offline rotation is fit: Q/K/V activations are captured
// offline and the rotation is derived from their covariance).
//
// Offline work, not on the decode path.  Three kernels on the caller's stream:
//   cov_kernel       Sigma += Q^T Q: CTA (i, j, c) accumulates the 64 x 64
//                    tile (i, j) of Sigma over row chunk c in float64 (a product
//                    of two float32 values is exact in float64; each thread a
//                    4 x 4 register block) and adds it into Sigma with float64
//                    atomics;
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
constexpr int kMaxSweeps = 40;
constexpr int kPairThreads = 256;

// Sigma tile (ti, tj) += Q^T Q over one chunk of rows; thread (ty, tx) owns a
// 4 x 4 block of the 64 x 64 tile; rows are staged as float64 (exact).
__global__ void __launch_bounds__(256) cov_kernel(const float* __restrict__ q, int64_t n, int D,
                                                  double* __restrict__ sigma) {
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
      sa[rr][cc] = in ? double(q[row * D + ti * kCovTile + cc]) : 0.0;
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
        if (ga != 0.0 && nrm > 0.0) {
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
                                double* __restrict__ lam, double* __restrict__ E, float* __restrict__ R, int D) {
  const int i = threadIdx.x;
  double n2 = 0.0;
  for (int r = 0; r < D; ++r) {
    const double a = A[int64_t(i) * D + r];
    n2 += a * a;
  }
  lam[i] = sqrt(n2);
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

}  // namespace

uint64_t calibrate_workspace_bytes(int D) { return 3 * align256(uint64_t(D) * D * 8) + align256(uint64_t(D) * 8) + 256; }

int launch_calibrate(const float* q, int64_t n, int D, float* R, void* ws, int32_t* status, cudaStream_t stream) {
  uint8_t* w = static_cast<uint8_t*>(ws);
  const uint64_t mat = align256(uint64_t(D) * D * 8);
  double* A = reinterpret_cast<double*>(w);  // Sigma, then Sigma V (columns)
  double* V = reinterpret_cast<double*>(w + mat);
  double* E = reinterpret_cast<double*>(w + 2 * mat);
  double* lam = reinterpret_cast<double*>(w + 3 * mat);
  unsigned long long* sweep_max = reinterpret_cast<unsigned long long*>(w + 3 * mat + align256(uint64_t(D) * 8));
  int32_t* info = reinterpret_cast<int32_t*>(sweep_max + 2);
  if (cudaMemsetAsync(A, 0, size_t(D) * D * 8, stream) != cudaSuccess) return OSCAR_ERR_LAUNCH;
  const int64_t chunks = (n + kCovChunk - 1) / kCovChunk;
  cov_kernel<<<dim3(D / kCovTile, D / kCovTile, unsigned(chunks)), 256, 0, stream>>>(q, n, D, A);
  if (cudaGetLastError() != cudaSuccess) return OSCAR_ERR_LAUNCH;
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
  finalize_kernel<<<1, D, 0, stream>>>(A, V, lam, E, R, D);
  return cudaGetLastError() == cudaSuccess ? OSCAR_OK : OSCAR_ERR_LAUNCH;
}

}  // namespace oscar
