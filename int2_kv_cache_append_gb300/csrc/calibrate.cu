// Calibration of the K-side rotation from query activations:
// Sigma = Q^T Q in float64, its eigenvectors by cyclic Jacobi in float64,
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
//   cov_kernel       Sigma += Q^T Q: CTA (i, j, c) accumulates the 32 x 32
//                    tile (i, j) of Sigma over row chunk c in float64 (a product
//                    of two float32 values is exact in float64) and adds it
//                    into Sigma with float64 atomics;
//   jacobi_kernel    one CTA: cyclic Jacobi in the round-robin ("circle")
//                    order, D/2 disjoint plane rotations per round applied
//                    together (rows, then columns and the eigenvector matrix),
//                    sweeps until the off-diagonal norm is below 1e-13 of the
//                    Frobenius norm, at most kMaxSweeps (then
//                    OSCAR_DEV_NOT_CONVERGED);
//   finalize_kernel  one CTA, one thread per eigenpair / row: rank the
//                    eigenvalues, move each eigenvector to its rank, sign it,
//                    apply H_D to every row with float64 butterflies and write
//                    column j of the result from column br(j), as float32.
#include <cuda_runtime.h>

#include "internal.h"

namespace oscar {
namespace {

constexpr int kCovTile = 32;
constexpr int kCovRows = 64;          // rows staged per step
constexpr int64_t kCovChunk = 4096;   // rows per CTA
constexpr int kMaxSweeps = 40;
constexpr int kJacobiThreads = 1024;

__global__ void __launch_bounds__(256) cov_kernel(const float* __restrict__ q, int64_t n, int D,
                                                  double* __restrict__ sigma) {
  __shared__ float ta[kCovRows][kCovTile + 1], tb[kCovRows][kCovTile + 1];
  const int ti = blockIdx.x, tj = blockIdx.y;
  const int t = threadIdx.x, r = t >> 3, c0 = (t & 7) * 4;
  const int64_t row_lo = int64_t(blockIdx.z) * kCovChunk;
  const int64_t row_hi = row_lo + kCovChunk < n ? row_lo + kCovChunk : n;
  double acc[4] = {0.0, 0.0, 0.0, 0.0};
  for (int64_t row0 = row_lo; row0 < row_hi; row0 += kCovRows) {
    for (int idx = t; idx < kCovRows * kCovTile; idx += 256) {
      const int rr = idx / kCovTile, cc = idx % kCovTile;
      const int64_t row = row0 + rr;
      const bool in = row < row_hi;
      ta[rr][cc] = in ? q[row * D + ti * kCovTile + cc] : 0.f;
      tb[rr][cc] = in ? q[row * D + tj * kCovTile + cc] : 0.f;
    }
    __syncthreads();
#pragma unroll 4
    for (int rr = 0; rr < kCovRows; ++rr) {
      const double a = double(ta[rr][r]);
#pragma unroll
      for (int m = 0; m < 4; ++m) acc[m] = fma(a, double(tb[rr][c0 + m]), acc[m]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int m = 0; m < 4; ++m) atomicAdd(&sigma[int64_t(ti * kCovTile + r) * D + tj * kCovTile + c0 + m], acc[m]);
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

__global__ void __launch_bounds__(kJacobiThreads) jacobi_kernel(double* __restrict__ A, double* __restrict__ V,
                                                                int D, int32_t* status, int32_t* info) {
  __shared__ double cs[256], sn[256];
  __shared__ int pp[256], qq[256];
  __shared__ double red[kJacobiThreads / 32];
  const int tid = threadIdx.x, nt = blockDim.x;
  const int64_t DD = int64_t(D) * D;
  for (int64_t idx = tid; idx < DD; idx += nt) V[idx] = (idx / D == idx % D) ? 1.0 : 0.0;
  __syncthreads();
  const int half = D / 2;
  int sweep = 0;
  bool converged = false;
  for (; sweep <= kMaxSweeps; ++sweep) {
    double off = 0.0, tot = 0.0;
    for (int64_t idx = tid; idx < DD; idx += nt) {
      const double a = A[idx];
      tot += a * a;
      if (idx / D != idx % D) off += a * a;
    }
    off = block_sum(off, red);
    tot = block_sum(tot, red);
    if (off <= 1e-26 * tot) {
      converged = true;
      break;
    }
    if (sweep == kMaxSweeps) break;
    for (int rnd = 0; rnd < D - 1; ++rnd) {
      // circle method: player D-1 fixed, players 0..D-2 rotate; pair k of
      // round rnd is (rnd, D-1) for k = 0, else (rnd + k, rnd - k) mod (D - 1)
      if (tid < half) {
        int p, q;
        if (tid == 0) {
          p = rnd;
          q = D - 1;
        } else {
          p = (rnd + tid) % (D - 1);
          q = (rnd - tid + (D - 1)) % (D - 1);
        }
        if (p > q) {
          const int x = p;
          p = q;
          q = x;
        }
        const double apq = A[int64_t(p) * D + q];
        double c = 1.0, s = 0.0;
        if (apq != 0.0) {
          // zero A[p][q]: tan of the angle is the smaller root of t^2 + 2 theta t - 1
          const double theta = (A[int64_t(q) * D + q] - A[int64_t(p) * D + p]) / (2.0 * apq);
          const double at = fabs(theta);
          const double tt = at > 1e150 ? 0.5 / at : 1.0 / (at + sqrt(theta * theta + 1.0));
          const double tv = theta < 0.0 ? -tt : tt;
          c = 1.0 / sqrt(tv * tv + 1.0);
          s = tv * c;
        }
        cs[tid] = c;
        sn[tid] = s;
        pp[tid] = p;
        qq[tid] = q;
      }
      __syncthreads();
      // rows p, q of A  (J^T A)
      for (int64_t idx = tid; idx < int64_t(half) * D; idx += nt) {
        const int k = int(idx / D), j = int(idx % D);
        const double c = cs[k], s = sn[k];
        double* rp = A + int64_t(pp[k]) * D + j;
        double* rq = A + int64_t(qq[k]) * D + j;
        const double ap = *rp, aq = *rq;
        *rp = c * ap - s * aq;
        *rq = s * ap + c * aq;
      }
      __syncthreads();
      // columns p, q of A and of V  (A J, V J)
      for (int64_t idx = tid; idx < int64_t(half) * D; idx += nt) {
        const int k = int(idx / D), i = int(idx % D);
        const double c = cs[k], s = sn[k];
        double* ap_ = A + int64_t(i) * D + pp[k];
        double* aq_ = A + int64_t(i) * D + qq[k];
        const double ap = *ap_, aq = *aq_;
        *ap_ = c * ap - s * aq;
        *aq_ = s * ap + c * aq;
        double* vp_ = V + int64_t(i) * D + pp[k];
        double* vq_ = V + int64_t(i) * D + qq[k];
        const double vp = *vp_, vq = *vq_;
        *vp_ = c * vp - s * vq;
        *vq_ = s * vp + c * vq;
      }
      __syncthreads();
    }
  }
  if (tid == 0) {
    info[0] = sweep;
    if (!converged) status_or(status, OSCAR_DEV_NOT_CONVERGED);
  }
}

__global__ void finalize_kernel(const double* __restrict__ A, const double* __restrict__ V, double* __restrict__ E,
                                float* __restrict__ R, int D) {
  const int i = threadIdx.x;  // eigenpair i, then column i, then row i
  const double li = A[int64_t(i) * D + i];
  int rank = 0;
  for (int j = 0; j < D; ++j) {
    const double lj = A[int64_t(j) * D + j];
    rank += (lj > li || (lj == li && j < i)) ? 1 : 0;
  }
  for (int r = 0; r < D; ++r) E[int64_t(r) * D + rank] = V[int64_t(r) * D + i];
  __syncthreads();
  // sign: the largest-magnitude entry of column i (the first, on ties) positive
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
  // row i times H_D: in-place Walsh-Hadamard butterflies, then 1/sqrt(D)
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

uint64_t calibrate_workspace_bytes(int D) { return 3 * align256(uint64_t(D) * D * 8) + 256; }

int launch_calibrate(const float* q, int64_t n, int D, float* R, void* ws, int32_t* status, cudaStream_t stream) {
  double* A = static_cast<double*>(ws);
  double* V = reinterpret_cast<double*>(static_cast<uint8_t*>(ws) + align256(uint64_t(D) * D * 8));
  double* E = reinterpret_cast<double*>(static_cast<uint8_t*>(ws) + 2 * align256(uint64_t(D) * D * 8));
  int32_t* info = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(ws) + 3 * align256(uint64_t(D) * D * 8));
  if (cudaMemsetAsync(A, 0, size_t(D) * D * 8, stream) != cudaSuccess) return OSCAR_ERR_LAUNCH;
  const int64_t chunks = (n + kCovChunk - 1) / kCovChunk;
  cov_kernel<<<dim3(D / kCovTile, D / kCovTile, unsigned(chunks)), 256, 0, stream>>>(q, n, D, A);
  if (cudaGetLastError() != cudaSuccess) return OSCAR_ERR_LAUNCH;
  jacobi_kernel<<<1, kJacobiThreads, 0, stream>>>(A, V, D, status, info);
  if (cudaGetLastError() != cudaSuccess) return OSCAR_ERR_LAUNCH;
  finalize_kernel<<<1, D, 0, stream>>>(A, V, E, R, D);
  return cudaGetLastError() == cudaSuccess ? OSCAR_OK : OSCAR_ERR_LAUNCH;
}

}  // namespace oscar
