// GPTQ on the GPU ("AWQ + GPTQ Quantization, in depth", section "The two
// algorithms, compactly"): H = 2 X X^T from calibration activations,
// H += damp * mean(diag H) * I, U = the upper Cholesky factor of H^-1, then
// columns in order (act order: by descending diag H), each rounded to its
// group's grid with the rounding error pushed onto the columns not yet
// quantized: W[:, j+1:] -= (w_j - q_j) / U[j, j] * U[j, j+1:].
//
// Everything is fp64 (the decisions that pick a code must match a fp64
// reference). Steps, one kernel family each:
//  1. gram_kernel: H = 2 x^T x.
//  2. prepare_kernel / rank_kernel: dead channels (diag 0 -> 1), damping,
//     the processing order (ranks by descending raw diag, ties to the lower
//     column) and the act-order group map.
//  3. A = J P^T H P J (P the processing order, J the index reversal), then
//     its lower Cholesky factor L (right-looking, 32-column panels), then
//     L^-1 (blocked). With H_p = P^T H P: J H_p J = L L^T gives
//     H_p^-1 = (J L^-1 J)^T (J L^-1 J), so U = J L^-1 J is upper triangular:
//     U[j][k] = L^-1[K-1-j][K-1-k].
//  4. gptq_kernel: every thread block owns 32 rows (rows are independent) and
//     walks the K columns in blocks of 32: the block's columns are updated in
//     shared memory one column at a time, and the columns after the block
//     take the block's errors at once (the page's "processing columns in
//     blocks"). A group's scale and zero point are set when its first column
//     is reached, from the current weights of its columns.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "internal.h"

namespace w4a16 {
namespace {

constexpr int NB = 32;  // panel / tile width

__global__ void __launch_bounds__(256) gram_kernel(const uint16_t* __restrict__ x, int64_t T, int K,
                                                   double* __restrict__ H) {
  __shared__ double xa[NB][NB + 1], xb[NB][NB + 1];
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // 32 x 8
  const int i0 = blockIdx.y * NB, j0 = blockIdx.x * NB;
  double acc[4] = {0, 0, 0, 0};
  for (int64_t t0 = 0; t0 < T; t0 += NB) {
    for (int r = ty; r < NB; r += 8) {
      const int64_t t = t0 + r;
      xa[r][tx] = (t < T && i0 + tx < K) ? double(__half2float(__ushort_as_half(x[t * K + i0 + tx]))) : 0.0;
      xb[r][tx] = (t < T && j0 + tx < K) ? double(__half2float(__ushort_as_half(x[t * K + j0 + tx]))) : 0.0;
    }
    __syncthreads();
#pragma unroll 8
    for (int r = 0; r < NB; ++r) {
      const double b = xb[r][tx];
#pragma unroll
      for (int u = 0; u < 4; ++u) acc[u] += xa[r][ty * 4 + u] * b;
    }
    __syncthreads();
  }
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int i = i0 + ty * 4 + u, j = j0 + tx;
    if (i < K && j < K) H[size_t(i) * K + j] = 2.0 * acc[u];
  }
}

// One block: raw diagonal into d, dead channels (diag 0: the channel never
// fires, its row and column are zero) get diag 1, then damp * mean(diag) is
// added to the diagonal.
__global__ void __launch_bounds__(1024) prepare_kernel(double* __restrict__ H, int K, double damp,
                                                       double* __restrict__ d) {
  __shared__ double part[1024];
  double s = 0.0;
  for (int i = threadIdx.x; i < K; i += blockDim.x) {
    double v = H[size_t(i) * K + i];
    d[i] = v;
    if (v == 0.0) {
      v = 1.0;
      H[size_t(i) * K + i] = 1.0;
    }
    s += v;
  }
  part[threadIdx.x] = s;
  __syncthreads();
  for (int o = blockDim.x / 2; o > 0; o >>= 1) {
    if (threadIdx.x < o) part[threadIdx.x] += part[threadIdx.x + o];
    __syncthreads();
  }
  const double lam = damp * part[0] / double(K);
  for (int i = threadIdx.x; i < K; i += blockDim.x) H[size_t(i) * K + i] += lam;
}

// order[rank] = column; g_idx[column] = rank / g (act order), else identity.
__global__ void __launch_bounds__(256) rank_kernel(const double* __restrict__ d, int K, int g, bool act,
                                                   int32_t* __restrict__ order, int32_t* __restrict__ g_idx) {
  const int j = blockIdx.x * blockDim.x + threadIdx.x;
  if (j >= K) return;
  int r = j;
  if (act) {
    const double dj = d[j];
    r = 0;
    for (int i = 0; i < K; ++i) {
      const double di = d[i];
      r += (di > dj || (di == dj && i < j)) ? 1 : 0;
    }
    g_idx[j] = r / g;
  }
  order[r] = j;
}

// A[a][b] = H[order[K-1-a]][order[K-1-b]], lower triangle only.
__global__ void __launch_bounds__(256) reverse_permute_kernel(const double* __restrict__ H, const int32_t* __restrict__ order,
                                                              int K, double* __restrict__ A) {
  const int64_t e = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (e >= int64_t(K) * K) return;
  const int a = int(e / K), b = int(e - int64_t(a) * K);
  if (b > a) return;
  A[e] = H[size_t(order[K - 1 - a]) * K + order[K - 1 - b]];
}

// ---- Cholesky, lower, in place: A = L L^T (32-column panels, right-looking)
__global__ void __launch_bounds__(NB) potrf_diag_kernel(double* __restrict__ A, int K, int k0) {
  __shared__ double s[NB][NB + 1];
  const int i = threadIdx.x;
  for (int c = 0; c < NB; ++c) s[i][c] = A[size_t(k0 + i) * K + k0 + c];
  __syncthreads();
  for (int c = 0; c < NB; ++c) {
    if (i == c) s[c][c] = sqrt(s[c][c]);
    __syncthreads();
    if (i > c) s[i][c] /= s[c][c];
    __syncthreads();
    if (i > c)
      for (int k = c + 1; k <= i; ++k) s[i][k] -= s[i][c] * s[k][c];
    __syncthreads();
  }
  for (int c = 0; c <= i; ++c) A[size_t(k0 + i) * K + k0 + c] = s[i][c];
}

// Rows below the panel: l = a L11^-T, i.e. L11 l^T = a^T (forward substitution).
__global__ void __launch_bounds__(128) trsm_kernel(double* __restrict__ A, int K, int k0) {
  __shared__ double L11[NB][NB + 1];
  for (int e = threadIdx.x; e < NB * NB; e += blockDim.x) {
    const int r = e / NB, c = e - r * NB;
    L11[r][c] = c <= r ? A[size_t(k0 + r) * K + k0 + c] : 0.0;
  }
  __syncthreads();
  const int i = k0 + NB + blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= K) return;
  double* row = A + size_t(i) * K + k0;
  double l[NB];
#pragma unroll
  for (int c = 0; c < NB; ++c) {
    double v = row[c];
#pragma unroll
    for (int k = 0; k < c; ++k) v -= L11[c][k] * l[k];
    l[c] = v / L11[c][c];
  }
#pragma unroll
  for (int c = 0; c < NB; ++c) row[c] = l[c];
}

// Trailing update of the lower triangle: A[i][j] -= sum_k L[i][k0+k] L[j][k0+k].
__global__ void __launch_bounds__(256) syrk_kernel(double* __restrict__ A, int K, int k0) {
  const int ti = blockIdx.y, tj = blockIdx.x;
  if (tj > ti) return;
  __shared__ double Pi[NB][NB + 1], Pj[NB][NB + 1];
  const int base = k0 + NB;
  const int i0 = base + ti * NB, j0 = base + tj * NB;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  for (int r = ty; r < NB; r += 8) {
    Pi[r][tx] = i0 + r < K ? A[size_t(i0 + r) * K + k0 + tx] : 0.0;
    Pj[r][tx] = j0 + r < K ? A[size_t(j0 + r) * K + k0 + tx] : 0.0;
  }
  __syncthreads();
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int ri = ty * 4 + u;
    const int i = i0 + ri, j = j0 + tx;
    if (i >= K || j >= K || j > i) continue;
    double acc = 0.0;
#pragma unroll 8
    for (int k = 0; k < NB; ++k) acc += Pi[ri][k] * Pj[tx][k];
    A[size_t(i) * K + j] -= acc;
  }
}

// ---- inverse of the lower triangular L (K a multiple of 32): diagonal blocks
// first, then block row by block row:
//   Linv[bi][bj] = -Linv[bi][bi] * sum_{bk = bj}^{bi-1} L[bi][bk] Linv[bk][bj]
__global__ void __launch_bounds__(NB) trinv_diag_kernel(const double* __restrict__ L, int K, double* __restrict__ Li) {
  __shared__ double s[NB][NB + 1];
  const int b0 = blockIdx.x * NB;
  const int c = threadIdx.x;  // this thread's column of the inverse
  for (int r = 0; r < NB; ++r) s[r][c] = c <= r ? L[size_t(b0 + r) * K + b0 + c] : 0.0;
  __syncthreads();
  double y[NB];
#pragma unroll
  for (int r = 0; r < NB; ++r) {
    double v = r == c ? 1.0 : 0.0;
#pragma unroll
    for (int k = 0; k < r; ++k) v -= s[r][k] * y[k];
    y[r] = r < c ? 0.0 : v / s[r][r];
  }
#pragma unroll
  for (int r = 0; r < NB; ++r) Li[size_t(b0 + r) * K + b0 + c] = y[r];
}

__global__ void __launch_bounds__(256) trinv_row_kernel(const double* __restrict__ L, int K, int bi,
                                                        double* __restrict__ Li) {
  const int bj = blockIdx.x;  // < bi
  __shared__ double Lt[NB][NB + 1], Xt[NB][NB + 1], T[NB][NB + 1];
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  double acc[4] = {0, 0, 0, 0};
  for (int bk = bj; bk < bi; ++bk) {
    for (int r = ty; r < NB; r += 8) {
      Lt[r][tx] = L[size_t(bi * NB + r) * K + bk * NB + tx];
      Xt[r][tx] = Li[size_t(bk * NB + r) * K + bj * NB + tx];
    }
    __syncthreads();
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int r = ty * 4 + u;
#pragma unroll 8
      for (int k = 0; k < NB; ++k) acc[u] += Lt[r][k] * Xt[k][tx];
    }
    __syncthreads();
  }
#pragma unroll
  for (int u = 0; u < 4; ++u) T[ty * 4 + u][tx] = acc[u];
  for (int r = ty; r < NB; r += 8) Lt[r][tx] = Li[size_t(bi * NB + r) * K + bi * NB + tx];  // Linv[bi][bi]
  __syncthreads();
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int r = ty * 4 + u;
    double v = 0.0;
#pragma unroll 8
    for (int k = 0; k < NB; ++k) v += Lt[r][k] * T[k][tx];
    Li[size_t(bi * NB + r) * K + bj * NB + tx] = -v;
  }
}

// Wp[n][j] = W[n][order[j]] (processing order, fp64).
__global__ void __launch_bounds__(256) load_weights_kernel(const uint16_t* __restrict__ w, const int32_t* __restrict__ order,
                                                           int64_t N, int K, double* __restrict__ Wp) {
  const int64_t e = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (e >= N * K) return;
  const int64_t n = e / K;
  const int j = int(e - n * K);
  Wp[e] = double(__half2float(__ushort_as_half(w[n * K + order[j]])));
}

struct GptqArgs {
  const double* Li;      // L^-1, U[j][k] = Li[K-1-j][K-1-k]
  const int32_t* order;  // processing position -> column
  double* Wp;            // N x K working weights, processing order
  uint8_t* q;            // N x K codes, original column order
  uint16_t* scales;      // N x G
  uint8_t* zeros;        // N x G or nullptr (symmetric)
  int64_t N;
  int K, g, bits;
  bool sym;
};

__device__ __forceinline__ double u_at(const GptqArgs& a, int j, int k) {
  return a.Li[size_t(a.K - 1 - j) * a.K + (a.K - 1 - k)];
}

__global__ void __launch_bounds__(256) gptq_kernel(const GptqArgs a) {
  __shared__ double Wb[NB][NB + 1];   // this block's rows x the current column block
  __shared__ double Ub[NB][NB + 1];   // U of the column block
  __shared__ double Er[NB][NB + 1];   // errors of the column block
  __shared__ double Ut[NB][2 * NB + 1];
  const int K = a.K, g = a.g;
  const int64_t r0 = int64_t(blockIdx.x) * NB;
  const int tid = threadIdx.x;
  const double qmax = double((1 << a.bits) - 1);
  const bool sym8 = a.sym && a.bits == 8;
  for (int j0 = 0; j0 < K; j0 += NB) {
    for (int e = tid; e < NB * NB; e += blockDim.x) {
      const int r = e / NB, c = e - r * NB;
      const int64_t n = r0 + r;
      Wb[r][c] = n < a.N ? a.Wp[n * K + j0 + c] : 0.0;
      Ub[r][c] = c >= r ? u_at(a, j0 + r, j0 + c) : 0.0;
    }
    __syncthreads();
    if (tid < NB && r0 + tid < a.N) {
      const int r = tid;
      const int64_t n = r0 + r;
      double s = 1.0, z = 0.0;
      for (int c = 0; c < NB; ++c) {
        const int j = j0 + c;
        if (j % g == 0 || c == 0) {
          // (group starts fall on column-block starts: g is a multiple of 32)
          const int t = j / g;
          if (j % g == 0) {
            double mn = INFINITY, mx = -INFINITY, am = 0.0;
            for (int cc = 0; cc < g; ++cc) {
              const double v = cc < NB ? Wb[r][cc] : a.Wp[n * K + j + cc];
              mn = fmin(mn, v);
              mx = fmax(mx, v);
              am = fmax(am, fabs(v));
            }
            const double range = a.sym ? (sym8 ? am / 127.0 : 2.0 * am / qmax) : (mx - mn) / qmax;
            __half sh = __double2half(range);
            if (__half2float(sh) == 0.0f) sh = __float2half(1.0f);
            s = double(__half2float(sh));
            z = a.sym ? double(1 << (a.bits - 1)) : fmin(fmax(rint(-mn / s), 0.0), qmax);
            a.scales[n * (K / g) + t] = __half_as_ushort(sh);
            if (a.zeros) a.zeros[n * (K / g) + t] = uint8_t(z);
          } else {
            // continuing a group that started in an earlier column block
            s = double(__half2float(__ushort_as_half(a.scales[n * (K / g) + t])));
            z = a.sym ? double(1 << (a.bits - 1)) : double(a.zeros[n * (K / g) + t]);
          }
        }
        const double w = Wb[r][c];
        double code;
        if (sym8) {
          code = fmin(fmax(rint(w / s), -127.0), 127.0) + 128.0;
        } else {
          code = fmin(fmax(rint(w / s) + z, 0.0), qmax);
        }
        const double wq = (code - z) * s;
        const double err = (w - wq) / Ub[c][c];
        Er[r][c] = err;
        for (int k = c + 1; k < NB; ++k) Wb[r][k] -= err * Ub[c][k];
        a.q[n * K + a.order[j]] = uint8_t(code);
      }
    }
    __syncthreads();
    // the columns after the block take the block's errors: Wp[:, ct..] -= Er * U[block, ct..]
    for (int ct = j0 + NB; ct < K; ct += 2 * NB) {
      for (int e = tid; e < NB * 2 * NB; e += blockDim.x) {
        const int r = e / (2 * NB), c = e - r * (2 * NB);
        Ut[r][c] = ct + c < K ? u_at(a, j0 + r, ct + c) : 0.0;
      }
      __syncthreads();
      for (int e = tid; e < NB * 2 * NB; e += blockDim.x) {
        const int r = e / (2 * NB), c = e - r * (2 * NB);
        const int64_t n = r0 + r;
        if (n < a.N && ct + c < K) {
          double acc = 0.0;
#pragma unroll 8
          for (int k = 0; k < NB; ++k) acc += Er[r][k] * Ut[k][c];
          a.Wp[n * K + ct + c] -= acc;
        }
      }
      __syncthreads();
    }
  }
}

inline unsigned blocks_for(int64_t n, int per) { return unsigned((n + per - 1) / per); }

}  // namespace

size_t gptq_workspace_bytes(int64_t N, int64_t K) {
  return align256(size_t(K) * K * 8) * 2 + align256(size_t(N) * K * 8) + align256(size_t(K) * 8) +
         align256(size_t(K) * 4);
}

cudaError_t launch_gptq(const Layout& L, const uint16_t* w, const uint16_t* x, int64_t T, double damp, uint8_t* q,
                        uint16_t* scales, uint8_t* zeros, int32_t* g_idx, void* workspace, cudaStream_t st) {
  const int K = int(L.K);
  const int64_t N = L.N;
  char* ws = static_cast<char*>(workspace);
  double* H = reinterpret_cast<double*>(ws);  // later L^-1
  ws += align256(size_t(K) * K * 8);
  double* A = reinterpret_cast<double*>(ws);  // reversed, permuted, damped H; then L
  ws += align256(size_t(K) * K * 8);
  double* Wp = reinterpret_cast<double*>(ws);
  ws += align256(size_t(N) * K * 8);
  double* d = reinterpret_cast<double*>(ws);
  ws += align256(size_t(K) * 8);
  int32_t* order = reinterpret_cast<int32_t*>(ws);

  const int tiles = (K + NB - 1) / NB;
  gram_kernel<<<dim3(tiles, tiles), 256, 0, st>>>(x, T, K, H);
  prepare_kernel<<<1, 1024, 0, st>>>(H, K, damp, d);
  rank_kernel<<<blocks_for(K, 256), 256, 0, st>>>(d, K, L.gsize, L.act, order, g_idx);
  reverse_permute_kernel<<<blocks_for(int64_t(K) * K, 256), 256, 0, st>>>(H, order, K, A);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  for (int k0 = 0; k0 < K; k0 += NB) {
    potrf_diag_kernel<<<1, NB, 0, st>>>(A, K, k0);
    const int rest = K - k0 - NB;
    if (rest > 0) {
      trsm_kernel<<<blocks_for(rest, 128), 128, 0, st>>>(A, K, k0);
      const int nt = (rest + NB - 1) / NB;
      syrk_kernel<<<dim3(nt, nt), 256, 0, st>>>(A, K, k0);
    }
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  double* Li = H;
  trinv_diag_kernel<<<K / NB, NB, 0, st>>>(A, K, Li);
  for (int bi = 1; bi < K / NB; ++bi) trinv_row_kernel<<<bi, 256, 0, st>>>(A, K, bi, Li);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  load_weights_kernel<<<blocks_for(N * K, 256), 256, 0, st>>>(w, order, N, K, Wp);
  GptqArgs a;
  a.Li = Li;
  a.order = order;
  a.Wp = Wp;
  a.q = q;
  a.scales = scales;
  a.zeros = L.sym ? nullptr : zeros;
  a.N = N;
  a.K = K;
  a.g = L.gsize;
  a.bits = L.bits;
  a.sym = L.sym;
  gptq_kernel<<<blocks_for(N, NB), 256, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace w4a16
