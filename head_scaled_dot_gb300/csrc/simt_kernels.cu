// simt_kernels.cu - CUDA-core (FMA) kernels for the fp32 path (and bf16 heads
// off the tensor cores): a tiled GEMM with the head-split / plain epilogue,
// and masked attention folded block by block with the stable summary
// (m, l, z) and its merge ("Stable summary of an attention key block",
// Definition, alphabetamath.cc), both register-tiled.
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

constexpr int TA_C = 64;  // keys per block

// 16 bytes from p (zeros when !ok; p is 16-byte aligned when ok).
__device__ __forceinline__ uint4 load16(const void* p, bool ok) {
  return ok ? *reinterpret_cast<const uint4*>(p) : make_uint4(0, 0, 0, 0);
}
// 16 bytes as floats: four fp32 or eight bf16 values.
__device__ __forceinline__ void unpack16(const uint4& a, float (&v)[4]) {
  v[0] = __uint_as_float(a.x);
  v[1] = __uint_as_float(a.y);
  v[2] = __uint_as_float(a.z);
  v[3] = __uint_as_float(a.w);
}
__device__ __forceinline__ void unpack16(const uint4& a, float (&v)[8]) {
  const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}
template <int VEC>
__device__ __forceinline__ void load_vec(const void* p, bool ok, float (&v)[VEC]) {
  unpack16(load16(p, ok), v);
}

struct AttnParams {
  const void* Q;
  const void* K;
  const void* V;
  void* Z;
  int n_q, n_k, h, d_h, d_vh;
  float c;
  int causal, padding, pad_queries;
  int vec_kv;  // K and V rows start on 16 bytes and hold whole 16-byte vectors
  int valid_len[MHA_MAX_PADDED_BATCH];
  int has_gate;                          // head_gate holds h entries (h <= MHA_MAX_GATED_HEADS)
  float head_gate[MHA_MAX_GATED_HEADS];  // per-head output scale, read only when has_gate
};

// grid (ceil(n_q / (16 RT)), h, B), 256 threads as 16 x 16 (ty, tx). A CTA
// folds the allowed keys of 16 RT query rows, 64 keys at a time, into each
// row's running summary (m, l, z), in base 2 (scores pre-multiplied by
// c log2(e)). Thread (ty, tx) holds the scores of rows RT ty + i and keys
// 4 tx + j (i < RT, j < 4), its share of each row's sum l, and z of rows
// RT ty + i, columns NV tx + j (j < NV; d_vh <= 16 NV). The row maximum of a
// block is taken across the 16 threads of a row (shuffles within a half
// warp); P goes through shared memory for z += P V. Register tiles keep a
// dozen or more FMAs per shared-memory load.
template <typename T, int NV, int RT>
__global__ void __launch_bounds__(256) attention_simt_kernel(const __grid_constant__ AttnParams P) {
  constexpr int DVP = 16 * NV;
  constexpr int TA_R = 16 * RT;  // query rows per CTA
  extern __shared__ float4 sm4[];
  float* sm = reinterpret_cast<float*>(sm4);
  const int dq = P.d_h, dv = P.d_vh;
  float* Qs = sm;                  // [dq][TA_R], scaled by c log2(e)
  float* Ks = Qs + dq * TA_R;      // [dq][TA_C]
  float* Vs = Ks + dq * TA_C;      // [TA_C][DVP], columns past d_vh zero
  float* Ps = Vs + TA_C * DVP;     // [TA_C][TA_R]
  const int b = blockIdx.z, head = blockIdx.y, q0 = blockIdx.x * TA_R;
  const int tid = threadIdx.x, ty = tid / 16, tx = tid % 16;
  const int L = P.padding ? P.valid_len[b] : P.n_k;
  const int q_end = P.pad_queries ? min(L, P.n_q) : P.n_q;
  const long long bh = (long long)b * P.h + head;
  const T* Qg = static_cast<const T*>(P.Q) + bh * P.n_q * dq;
  const T* Kg = static_cast<const T*>(P.K) + bh * P.n_k * dq;
  const T* Vg = static_cast<const T*>(P.V) + bh * P.n_k * dv;
  T* Zg = static_cast<T*>(P.Z);
  const float cl2 = P.c * 1.4426950408889634f;

  for (int e = tid; e < TA_R * dq; e += 256) {
    const int r = e % TA_R, k = e / TA_R;
    Qs[e] = (q0 + r < P.n_q) ? to_f(Qg[(long long)(q0 + r) * dq + k]) * cl2 : 0.f;
  }
  // Keys this CTA can use: [0, k_end). Rows of K and V at or past L are never
  // read (loaded as zeros), so they may hold anything.
  int k_end = L;
  if (P.causal) k_end = min(k_end, q0 + TA_R);

  float m_run[RT], l_run[RT], z[RT][NV];
#pragma unroll
  for (int i = 0; i < RT; ++i) {
    m_run[i] = -INFINITY;
    l_run[i] = 0.f;
#pragma unroll
    for (int j = 0; j < NV; ++j) z[i][j] = 0.f;
  }

  // 16-byte loads of K and V rows when every row starts on 16 bytes. When a
  // block's K and V are at most 256 vectors each (bf16 heads up to 32, fp32
  // up to 16), each thread loads its vector of the next block into registers
  // while the current block is computed and stores it to shared memory at
  // the top of the next block, so the loads' latency is not waited for.
  constexpr int VEC = 16 / sizeof(T);
  const bool vec = P.vec_kv;
  const int kvec = dq / VEC, vvec = DVP / VEC;
  const bool ahead = vec && TA_C * kvec <= 256 && TA_C * vvec <= 256;
  uint4 kreg = make_uint4(0, 0, 0, 0), vreg = make_uint4(0, 0, 0, 0);
  auto fetch = [&](int kb) {
    if (tid < TA_C * kvec) {
      const int c = tid / kvec, k = (tid % kvec) * VEC;
      kreg = load16(Kg + (long long)(kb + c) * dq + k, kb + c < L);
    }
    if (tid < TA_C * vvec) {
      const int c = tid / vvec, col = (tid % vvec) * VEC;
      vreg = load16(Vg + (long long)(kb + c) * dv + col, kb + c < L && col < dv);
    }
  };
  if (ahead && k_end > 0) fetch(0);
  for (int k0 = 0; k0 < k_end; k0 += TA_C) {
    __syncthreads();  // the previous block's K, V and P are no longer read
    if (ahead) {
      if (tid < TA_C * kvec) {
        const int c = tid / kvec, k = (tid % kvec) * VEC;
        float v[VEC];
        unpack16(kreg, v);
#pragma unroll
        for (int u = 0; u < VEC; ++u) Ks[(k + u) * TA_C + c] = v[u];
      }
      if (tid < TA_C * vvec) {
        const int c = tid / vvec, col = (tid % vvec) * VEC;
        float v[VEC];
        unpack16(vreg, v);
#pragma unroll
        for (int u = 0; u < VEC; ++u) Vs[c * DVP + col + u] = v[u];
      }
      if (k0 + TA_C < k_end) fetch(k0 + TA_C);
    } else if (vec) {
      for (int e = tid; e < TA_C * (dq / VEC); e += 256) {
        const int c = e / (dq / VEC), k = (e % (dq / VEC)) * VEC;
        float v[VEC];
        load_vec(Kg + (long long)(k0 + c) * dq + k, k0 + c < L, v);
#pragma unroll
        for (int u = 0; u < VEC; ++u) Ks[(k + u) * TA_C + c] = v[u];
      }
      for (int e = tid; e < TA_C * (DVP / VEC); e += 256) {
        const int c = e / (DVP / VEC), col = (e % (DVP / VEC)) * VEC;
        float v[VEC];
        load_vec(Vg + (long long)(k0 + c) * dv + col, k0 + c < L && col < dv, v);
#pragma unroll
        for (int u = 0; u < VEC; ++u) Vs[c * DVP + col + u] = v[u];
      }
    } else {
      for (int e = tid; e < TA_C * dq; e += 256) {
        const int c = e % TA_C, k = e / TA_C;
        Ks[e] = (k0 + c < L) ? to_f(Kg[(long long)(k0 + c) * dq + k]) : 0.f;
      }
      for (int e = tid; e < TA_C * DVP; e += 256) {
        const int c = e / DVP, col = e % DVP;
        Vs[e] = (k0 + c < L && col < dv) ? to_f(Vg[(long long)(k0 + c) * dv + col]) : 0.f;
      }
    }
    __syncthreads();
    // scores of this thread's 4 x 4 tile
    float s[RT][4];
#pragma unroll
    for (int i = 0; i < RT; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) s[i][j] = 0.f;
#pragma unroll 4
    for (int k = 0; k < dq; ++k) {
      float qa[RT];
#pragma unroll
      for (int i4 = 0; i4 < RT; i4 += 4) {
        const float4 qv = *reinterpret_cast<const float4*>(Qs + k * TA_R + RT * ty + i4);
        qa[i4] = qv.x;
        qa[i4 + 1] = qv.y;
        qa[i4 + 2] = qv.z;
        qa[i4 + 3] = qv.w;
      }
      const float4 kv = *reinterpret_cast<const float4*>(Ks + k * TA_C + 4 * tx);
      const float ka[4] = {kv.x, kv.y, kv.z, kv.w};
#pragma unroll
      for (int i = 0; i < RT; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) s[i][j] = fmaf(qa[i], ka[j], s[i][j]);
    }
    // fold the block into each row's summary
    float pcol[RT][4];  // p of key 4 tx + j, row RT ty + i
#pragma unroll
    for (int i = 0; i < RT; ++i) {
      const int q = q0 + RT * ty + i;
      float mb = -INFINITY;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int key = k0 + 4 * tx + j;
        const bool allowed = key < L && (!P.causal || key <= q);
        if (!allowed) s[i][j] = -INFINITY;  // weight exactly 0
        mb = fmaxf(mb, s[i][j]);
      }
#pragma unroll
      for (int o = 1; o < 16; o <<= 1) mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, o));
      const float m_new = fmaxf(m_run[i], mb);
      // e^{m - m'} (1 when m is kept, also while the row has no allowed key yet)
      const float a = (m_new == m_run[i]) ? 1.f : ex2_approx(m_run[i] - m_new);
      float ls = 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float p = (s[i][j] == -INFINITY) ? 0.f : ex2_approx(s[i][j] - m_new);
        pcol[i][j] = p;
        ls += p;
      }
      l_run[i] = l_run[i] * a + ls;
#pragma unroll
      for (int j = 0; j < NV; ++j) z[i][j] *= a;
      m_run[i] = m_new;
    }
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int i4 = 0; i4 < RT; i4 += 4)
        *reinterpret_cast<float4*>(Ps + (4 * tx + j) * TA_R + RT * ty + i4) =
            make_float4(pcol[i4][j], pcol[i4 + 1][j], pcol[i4 + 2][j], pcol[i4 + 3][j]);
    __syncthreads();
    // z += P V over the block's keys
    const int nc = min(TA_C, k_end - k0);
#pragma unroll 4
    for (int c = 0; c < nc; ++c) {
      float pa[RT];
#pragma unroll
      for (int i4 = 0; i4 < RT; i4 += 4) {
        const float4 pv = *reinterpret_cast<const float4*>(Ps + c * TA_R + RT * ty + i4);
        pa[i4] = pv.x;
        pa[i4 + 1] = pv.y;
        pa[i4 + 2] = pv.z;
        pa[i4 + 3] = pv.w;
      }
      // this thread's NV adjacent columns of V row c, in one to four loads
      float va[NV];
      const float* vrow = Vs + c * DVP + NV * tx;
      if constexpr (NV == 1) {
        va[0] = vrow[0];
      } else if constexpr (NV == 2) {
        const float2 t2 = *reinterpret_cast<const float2*>(vrow);
        va[0] = t2.x;
        va[1] = t2.y;
      } else {
#pragma unroll
        for (int j4 = 0; j4 < NV; j4 += 4) {
          const float4 t4 = *reinterpret_cast<const float4*>(vrow + j4);
          va[j4] = t4.x;
          va[j4 + 1] = t4.y;
          va[j4 + 2] = t4.z;
          va[j4 + 3] = t4.w;
        }
      }
#pragma unroll
      for (int j = 0; j < NV; ++j)
#pragma unroll
        for (int i = 0; i < RT; ++i) z[i][j] = fmaf(pa[i], va[j], z[i][j]);
    }
  }
  // the row sum is spread over the row's 16 threads
#pragma unroll
  for (int i = 0; i < RT; ++i)
#pragma unroll
    for (int o = 1; o < 16; o <<= 1) l_run[i] += __shfl_xor_sync(0xffffffffu, l_run[i], o);
#pragma unroll
  for (int i = 0; i < RT; ++i) {
    const int q = q0 + RT * ty + i;
    if (q >= P.n_q) continue;
    const bool computed = q < q_end;
    const float inv = computed ? (P.has_gate ? P.head_gate[head] : 1.f) / l_run[i] : 0.f;
    T* zrow = Zg + ((long long)b * P.n_q + q) * (long long)P.h * dv + (long long)head * dv;
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      const int col = NV * tx + j;
      if (col < dv) zrow[col] = from_f<T>(computed ? z[i][j] * inv : 0.f);
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

template <typename T, int NV, int RT>
mha_status launch_attention_simt(const AttnParams& P, int B, cudaStream_t s) {
  constexpr int TA_R = 16 * RT;
  const dim3 grid((P.n_q + TA_R - 1) / TA_R, P.h, B);
  if (grid.y > 65535u || grid.z > 65535u) return MHA_ERR_UNSUPPORTED;
  const size_t smem =
      sizeof(float) * ((size_t)P.d_h * (TA_R + TA_C) + (size_t)TA_C * 16 * NV + TA_C * TA_R);
  if (!ensure_smem_limit((const void*)attention_simt_kernel<T, NV, RT>, (int)smem))
    return MHA_ERR_CUDA;
  attention_simt_kernel<T, NV, RT><<<grid, 256, smem, s>>>(P);
  count_launch();
  return cudaGetLastError() == cudaSuccess ? MHA_OK : MHA_ERR_CUDA;
}

// Narrow value heads take 8 query rows per thread (more FMAs per shared
// load) when that still leaves two CTAs per SM, wide ones 4 (registers for z).
template <typename T>
mha_status launch_attention_simt_dv(const AttnParams& P, int B, cudaStream_t s) {
  const bool tall = (long long)((P.n_q + 127) / 128) * P.h * B >= 2LL * num_sms();
  if (P.d_vh <= 16)
    return tall ? launch_attention_simt<T, 1, 8>(P, B, s) : launch_attention_simt<T, 1, 4>(P, B, s);
  if (P.d_vh <= 32)
    return tall ? launch_attention_simt<T, 2, 8>(P, B, s) : launch_attention_simt<T, 2, 4>(P, B, s);
  if (P.d_vh <= 64)
    return tall ? launch_attention_simt<T, 4, 8>(P, B, s) : launch_attention_simt<T, 4, 4>(P, B, s);
  if (P.d_vh <= 128) return launch_attention_simt<T, 8, 4>(P, B, s);
  return launch_attention_simt<T, 16, 4>(P, B, s);
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
  {
    const int vec = dt == MHA_DTYPE_F32 ? 4 : 8;  // elements per 16 bytes
    auto al16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    P.vec_kv = a.d_h % vec == 0 && a.d_vh % vec == 0 && al16(a.K) && al16(a.V);
  }
  for (int b = 0; b < MHA_MAX_PADDED_BATCH; ++b)
    P.valid_len[b] = (a.padding && b < a.B) ? a.valid_len_host[b] : a.n_k;
  P.has_gate = a.head_gate_host != nullptr && a.h <= MHA_MAX_GATED_HEADS;
  for (int i = 0; i < MHA_MAX_GATED_HEADS; ++i)
    P.head_gate[i] = (P.has_gate && i < a.h) ? a.head_gate_host[i] : 1.f;
  if (dt == MHA_DTYPE_F32) return launch_attention_simt_dv<float>(P, a.B, s);
  return launch_attention_simt_dv<__nv_bfloat16>(P, a.B, s);
}

}  // namespace mha
