// simt_kernels.cu - CUDA-core (FMA) kernels for the fp32 path: a tiled GEMM
// with the head-split / plain epilogue, and masked attention folded block by
// block with the stable summary (m, l, z) and its merge ("Stable summary of
// an attention key block", Definition, alphabetamath.cc).
//
// fp32 inputs keep 1e-4 relative accuracy here, which tf32 tensor cores
// (10-bit mantissa) cannot; these kernels are the fp32 compute path.
#include <cuda_bf16.h>
#include <math.h>

#include "device_common.cuh"
#include "internal.h"

namespace mha {
namespace {

template <typename T>
__device__ __forceinline__ float to_f(T x);
template <>
__device__ __forceinline__ float to_f<float>(float x) {
  return x;
}
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) {
  return __bfloat162float(x);
}

template <typename T>
__device__ __forceinline__ T from_f(float x);
template <>
__device__ __forceinline__ float from_f<float>(float x) {
  return x;
}
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

struct GemmBatch {
  GemmProblem p[3];
};

constexpr int GT_M = 64, GT_N = 64, GT_K = 16;

// 256 threads, one 64 x 64 output tile per CTA, 4 x 4 outputs per thread.
// blockIdx.z selects the problem of the grouped launch.
template <typename T>
__global__ void __launch_bounds__(256) gemm_simt_kernel(const __grid_constant__ GemmBatch batch) {
  const GemmProblem& P = batch.p[blockIdx.z];
  const int m0 = blockIdx.y * GT_M, n0 = blockIdx.x * GT_N;
  if (m0 >= P.M || n0 >= P.N) return;
  __shared__ float As[GT_K][GT_M + 4];
  __shared__ float Ws[GT_K][GT_N + 4];
  const T* A = static_cast<const T*>(P.A);
  const T* W = static_cast<const T*>(P.W);
  const int tid = threadIdx.x;
  const int tr = tid / 16, tc = tid % 16;  // 16 x 16 threads, 4 x 4 each
  float acc[4][4] = {};
  for (int k0 = 0; k0 < P.K; k0 += GT_K) {
    for (int e = tid; e < GT_M * GT_K; e += 256) {
      const int r = e / GT_K, k = e % GT_K;
      const int m = m0 + r, kk = k0 + k;
      As[k][r] = (m < P.M && kk < P.K) ? to_f(A[(long long)m * P.K + kk]) : 0.f;
    }
    for (int e = tid; e < GT_K * GT_N; e += 256) {
      const int k = e / GT_N, c = e % GT_N;
      const int n = n0 + c, kk = k0 + k;
      Ws[k][c] = (n < P.N && kk < P.K) ? to_f(W[(long long)kk * P.N + n]) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < GT_K; ++k) {
      float a[4], w[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[k][tr * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) w[j] = Ws[k][tc * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], w[j], acc[i][j]);
    }
    __syncthreads();
  }
  T* out = static_cast<T*>(P.out);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = m0 + tr * 4 + i;
    if (m >= P.M) continue;
    const long long row_off =
        (long long)(m / P.rows_per_group) * P.s_group_row + (long long)(m % P.rows_per_group) * P.s_row;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tc * 4 + j;
      if (n >= P.N) continue;
      const long long off = row_off + (long long)(n / P.cols_per_group) * P.s_group_col +
                            (n % P.cols_per_group);
      out[off] = from_f<T>(acc[i][j]);
    }
  }
}

constexpr int AT_ROWS = 32;  // query rows per CTA (4 per warp)
constexpr int AT_KEYS = 32;  // keys per block (one per lane)

struct AttnParams {
  const void* Q;
  const void* K;
  const void* V;
  void* Z;
  int n_q, n_k, h, d_h, d_vh;
  float c;
  int causal, padding, pad_queries;
  int valid_len[MHA_MAX_PADDED_BATCH];
  int has_gate;                          // head_gate holds h entries (h <= MHA_MAX_GATED_HEADS)
  float head_gate[MHA_MAX_GATED_HEADS];  // per-head output scale, read only when has_gate
};

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// grid (ceil(n_q / 32), h, B), 256 threads. Lane j of a warp scores key j of
// the current 32-key block for one query row; the block's summary
// (m_blk, l_blk, z_blk) is merged into the row's running summary. Head sizes
// up to AT_DMAX (d_vh columns: lane + 32 t).
template <typename T, int AT_DMAX>
__global__ void __launch_bounds__(256) attention_simt_kernel(const __grid_constant__ AttnParams P) {
  extern __shared__ float sm[];
  const int dq = P.d_h, dv = P.d_vh;
  float* Qs = sm;                       // [AT_ROWS][dq]
  float* Ks = Qs + AT_ROWS * dq;        // [AT_KEYS][dq + 1]
  float* Vs = Ks + AT_KEYS * (dq + 1);  // [AT_KEYS][dv]
  const int b = blockIdx.z, head = blockIdx.y, q0 = blockIdx.x * AT_ROWS;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int L = P.padding ? P.valid_len[b] : P.n_k;
  const int q_end = P.pad_queries ? min(L, P.n_q) : P.n_q;
  const long long bh = (long long)b * P.h + head;
  const T* Qg = static_cast<const T*>(P.Q) + bh * P.n_q * dq;
  const T* Kg = static_cast<const T*>(P.K) + bh * P.n_k * dq;
  const T* Vg = static_cast<const T*>(P.V) + bh * P.n_k * dv;
  T* Zg = static_cast<T*>(P.Z);

  for (int e = threadIdx.x; e < AT_ROWS * dq; e += blockDim.x) {
    const int r = e / dq, k = e % dq;
    Qs[e] = (q0 + r < P.n_q) ? to_f(Qg[(long long)(q0 + r) * dq + k]) : 0.f;
  }
  // Keys this CTA can use: [0, k_end). Rows of K and V at or past L are never
  // read (loaded as zeros), so they may hold anything.
  int k_end = L;
  if (P.causal) k_end = min(k_end, q0 + AT_ROWS);

  float m_run[4], l_run[4], z_run[4][AT_DMAX / 32];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    m_run[i] = -INFINITY;
    l_run[i] = 0.f;
#pragma unroll
    for (int t = 0; t < AT_DMAX / 32; ++t) z_run[i][t] = 0.f;
  }

  for (int k0 = 0; k0 < k_end; k0 += AT_KEYS) {
    __syncthreads();
    for (int e = threadIdx.x; e < AT_KEYS * dq; e += blockDim.x) {
      const int j = e / dq, k = e % dq;
      Ks[j * (dq + 1) + k] = (k0 + j < L) ? to_f(Kg[(long long)(k0 + j) * dq + k]) : 0.f;
    }
    for (int e = threadIdx.x; e < AT_KEYS * dv; e += blockDim.x) {
      const int j = e / dv, k = e % dv;
      Vs[e] = (k0 + j < L) ? to_f(Vg[(long long)(k0 + j) * dv + k]) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = warp * 4 + i, q = q0 + r;
      if (q >= q_end) continue;  // warp-uniform
      const int key = k0 + lane;
      const bool allowed = key < L && (!P.causal || key <= q);
      float s = 0.f;
      for (int k = 0; k < dq; ++k) s = fmaf(Qs[r * dq + k], Ks[lane * (dq + 1) + k], s);
      s *= P.c;
      const float m_blk = warp_max(allowed ? s : -INFINITY);
      if (m_blk == -INFINITY) continue;  // empty block: the bottom summary
      const float p = allowed ? expf(s - m_blk) : 0.f;
      const float l_blk = warp_sum(p);
      float z_blk[AT_DMAX / 32];
#pragma unroll
      for (int t = 0; t < AT_DMAX / 32; ++t) z_blk[t] = 0.f;
      for (int j = 0; j < AT_KEYS; ++j) {
        const float pj = __shfl_sync(0xffffffffu, p, j);
#pragma unroll
        for (int t = 0; t < AT_DMAX / 32; ++t) {
          const int col = lane + 32 * t;
          if (col < dv) z_blk[t] = fmaf(pj, Vs[j * dv + col], z_blk[t]);
        }
      }
      // merge: m' = max(m_S, m_T); scale each side by e^{m - m'}
      const float m_new = fmaxf(m_run[i], m_blk);
      const float a = expf(m_run[i] - m_new), bsc = expf(m_blk - m_new);
      l_run[i] = a * l_run[i] + bsc * l_blk;
#pragma unroll
      for (int t = 0; t < AT_DMAX / 32; ++t) z_run[i][t] = a * z_run[i][t] + bsc * z_blk[t];
      m_run[i] = m_new;
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int q = q0 + warp * 4 + i;
    if (q >= P.n_q) continue;
    const bool computed = q < q_end;
    const float inv = computed ? (P.has_gate ? P.head_gate[head] : 1.f) / l_run[i] : 0.f;
    T* zrow = Zg + ((long long)b * P.n_q + q) * (long long)P.h * dv + (long long)head * dv;
#pragma unroll
    for (int t = 0; t < AT_DMAX / 32; ++t) {
      const int col = lane + 32 * t;
      if (col < dv) zrow[col] = from_f<T>(computed ? z_run[i][t] * inv : 0.f);
    }
  }
}

}  // namespace

mha_status gemm_simt(const GemmProblem* probs, int nprob, mha_dtype dt, cudaStream_t s) {
  GemmBatch batch{};
  int max_m = 0, max_n = 0;
  for (int i = 0; i < nprob; ++i) {
    batch.p[i] = probs[i];
    max_m = max(max_m, probs[i].M);
    max_n = max(max_n, probs[i].N);
  }
  const dim3 grid((max_n + GT_N - 1) / GT_N, (max_m + GT_M - 1) / GT_M, nprob);
  if (grid.y > 65535u) return MHA_ERR_UNSUPPORTED;
  if (dt == MHA_DTYPE_F32)
    gemm_simt_kernel<float><<<grid, 256, 0, s>>>(batch);
  else
    gemm_simt_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(batch);
  count_launch();
  return cudaGetLastError() == cudaSuccess ? MHA_OK : MHA_ERR_CUDA;
}

namespace {

template <typename T, int DMAX>
mha_status launch_attention_simt(const AttnParams& P, const dim3& grid, size_t smem,
                                 cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(attention_simt_kernel<T, DMAX>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return MHA_ERR_CUDA;
  attention_simt_kernel<T, DMAX><<<grid, 256, smem, s>>>(P);
  count_launch();
  return cudaGetLastError() == cudaSuccess ? MHA_OK : MHA_ERR_CUDA;
}

}  // namespace

mha_status attention_simt(const AttnArgs& a, mha_dtype dt, cudaStream_t s) {
  if (a.d_h > 256 || a.d_vh > 256) return MHA_ERR_UNSUPPORTED;
  AttnParams P;
  P.Q = a.Q;
  P.K = a.K;
  P.V = a.V;
  P.Z = a.Z;
  P.n_q = a.n_q;
  P.n_k = a.n_k;
  P.h = a.h;
  P.d_h = a.d_h;
  P.d_vh = a.d_vh;
  P.c = a.c;
  P.causal = a.causal;
  P.padding = a.padding;
  P.pad_queries = a.pad_queries;
  for (int b = 0; b < MHA_MAX_PADDED_BATCH; ++b)
    P.valid_len[b] = (a.padding && b < a.B) ? a.valid_len_host[b] : a.n_k;
  P.has_gate = a.head_gate_host != nullptr && a.h <= MHA_MAX_GATED_HEADS;
  for (int i = 0; i < MHA_MAX_GATED_HEADS; ++i)
    P.head_gate[i] = (P.has_gate && i < a.h) ? a.head_gate_host[i] : 1.f;
  const size_t smem =
      sizeof(float) * (AT_ROWS * a.d_h + AT_KEYS * (a.d_h + 1) + AT_KEYS * a.d_vh);
  const dim3 grid((a.n_q + AT_ROWS - 1) / AT_ROWS, a.h, a.B);
  if (grid.y > 65535u || grid.z > 65535u) return MHA_ERR_UNSUPPORTED;
  const bool wide = a.d_vh > 128;
  if (dt == MHA_DTYPE_F32)
    return wide ? launch_attention_simt<float, 256>(P, grid, smem, s)
                : launch_attention_simt<float, 128>(P, grid, smem, s);
  return wide ? launch_attention_simt<__nv_bfloat16, 256>(P, grid, smem, s)
              : launch_attention_simt<__nv_bfloat16, 128>(P, grid, smem, s);
}

}  // namespace mha
