// mha_api.cu - the C ABI (include/mha.h): argument checks, workspace layout,
// dispatch of the three steps, device error word, TMA descriptor encoding.
#include <cudaTypedefs.h>
#include <math.h>
#include <stdio.h>
#include <string.h>

#include <atomic>
#include <mutex>
#include <vector>

#include "device_common.cuh"
#include "internal.h"

namespace mha {

static std::atomic<uint64_t> g_launches{0};

void count_launch(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

// Bounded waits give up after this long. Long enough for any legitimate wait
// (a whole kernel takes milliseconds), short enough to free a shared GPU fast.
uint64_t wait_limit_ns() { return 2000000000ull; }

// Streaming multiprocessors of the current device (persistent grids).
int num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    return 148;
  return n;
}

// Per-device kernel set-up, cached under one lock.
namespace {
struct KernelSetup {
  const void* kernel;
  int dev;
  int smem_limit;  // dynamic shared memory raised to this (0: not set)
  int resident;    // CTAs per SM (0: not asked)
};
std::mutex g_setup_mu;
std::vector<KernelSetup> g_setup;

KernelSetup* find_setup(const void* kernel, int dev) {
  for (auto& k : g_setup)
    if (k.kernel == kernel && k.dev == dev) return &k;
  g_setup.push_back({kernel, dev, 0, 0});
  return &g_setup.back();
}
}  // namespace

bool ensure_smem_limit(const void* kernel, int bytes) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  std::lock_guard<std::mutex> lock(g_setup_mu);
  KernelSetup* k = find_setup(kernel, dev);
  if (k->smem_limit >= bytes) return true;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) !=
      cudaSuccess)
    return false;
  k->smem_limit = bytes;
  return true;
}

int resident_ctas(const void* kernel, int threads, int smem_bytes) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  std::lock_guard<std::mutex> lock(g_setup_mu);
  KernelSetup* k = find_setup(kernel, dev);
  if (k->resident < 1) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, smem_bytes) !=
            cudaSuccess ||
        n < 1)
      n = 1;
    k->resident = n;
  }
  return k->resident;
}

// ---------------------------------------------------------------------------
// TMA descriptors
// ---------------------------------------------------------------------------

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

bool make_tmap_bf16(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                    const uint64_t* strides_bytes, const uint32_t* box, bool swizzle128) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t d[5], st[4];
  cuuint32_t bx[5], es[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    bx[i] = box[i];
    es[i] = 1;
    if (i + 1 < rank) st[i] = strides_bytes[i];
  }
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank, const_cast<void*>(base),
                  d, st, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// ---------------------------------------------------------------------------
// Failure-detection self-test kernel
// ---------------------------------------------------------------------------

__global__ void selftest_wait_kernel(int32_t* err, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar, 1);  // one arrival expected; nothing ever arrives
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    WaitCtl w{err, &abort_flag, limit_ns};
    mbar_wait(&bar, 0, w);
  }
  __syncthreads();
}

mha_status selftest_wait(int32_t* err, uint64_t limit_ns, cudaStream_t s) {
  selftest_wait_kernel<<<1, 32, 0, s>>>(err, limit_ns);
  count_launch();
  return cudaGetLastError() == cudaSuccess ? MHA_OK : MHA_ERR_CUDA;
}

}  // namespace mha

using namespace mha;

namespace {

constexpr size_t kHeader = 256;

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

size_t elem_size(mha_dtype dt) { return dt == MHA_DTYPE_F32 ? 4 : 2; }

bool dtype_ok(mha_dtype dt) { return dt == MHA_DTYPE_F32 || dt == MHA_DTYPE_BF16; }

bool mask_ok(mha_mask_kind m) {
  return m == MHA_MASK_NONE || m == MHA_MASK_CAUSAL || m == MHA_MASK_PADDING ||
         m == MHA_MASK_CAUSAL_PADDING;
}

bool has_causal(mha_mask_kind m) { return m == MHA_MASK_CAUSAL || m == MHA_MASK_CAUSAL_PADDING; }
bool has_padding(mha_mask_kind m) {
  return m == MHA_MASK_PADDING || m == MHA_MASK_CAUSAL_PADDING;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool tc_head_dims(int d_h, int d_vh);

struct Layout {
  size_t q, k, v, z, split, split_bytes, total;
};

// Error word, Q, K, V, Z, then the scratch of the automatic split over the
// keys (bf16 heads on the tensor cores whose tile pairs leave SMs idle).
Layout layout(int B, int n_q, int n_k, int h, int d_h, int d_vh, mha_dtype dt) {
  const size_t es = elem_size(dt);
  Layout L;
  L.q = kHeader;
  L.k = align_up(L.q + (size_t)B * h * n_q * d_h * es, 1024);
  L.v = align_up(L.k + (size_t)B * h * n_k * d_h * es, 1024);
  L.z = align_up(L.v + (size_t)B * h * n_k * d_vh * es, 1024);
  L.split = align_up(L.z + (size_t)B * n_q * h * d_vh * es, 1024);
  L.split_bytes = (dt == MHA_DTYPE_BF16 && tc_head_dims(d_h, d_vh))
                      ? attention_auto_split_bytes(B, n_q, n_k, h, d_vh)
                      : 0;
  L.total = align_up(L.split + L.split_bytes, 1024);
  return L;
}

// Head sizes every path handles: 1 .. MAX_HEAD_DIM. bf16 heads of 32..128
// (multiples of 8) run on the tensor cores, other sizes on the CUDA-core
// kernel.
constexpr int MAX_HEAD_DIM = 256;

mha_status check_head_dims(int d_h, int d_vh, mha_dtype dt) {
  (void)dt;
  if (d_h > MAX_HEAD_DIM || d_vh > MAX_HEAD_DIM) return MHA_ERR_UNSUPPORTED;
  return MHA_OK;
}

// Head sizes the tensor-core attention kernels take: 64, or 72..128 run in
// the 128-wide kernels (multiples of 8, as their tensor maps need 16-byte
// strides).
bool tc_head_dims(int d_h, int d_vh) {
  auto ok = [](int d) { return d >= 32 && d <= 128 && d % 8 == 0; };
  return ok(d_h) && ok(d_vh);
}

// Elements beyond 2^31 per tensor are not addressed by every index path.
bool fits(long long a, long long b, long long c) {
  const long long lim = (1ll << 31) - 1;
  return a > 0 && b > 0 && c > 0 && a <= lim / b && a * b <= lim / c;
}

mha_status check_valid_len(mha_mask_kind mask, const int32_t* valid_len, int B, int n_k) {
  if (!has_padding(mask)) return MHA_OK;
  if (!valid_len) return MHA_ERR_INVALID_ARG;
  if (B > MHA_MAX_PADDED_BATCH) return MHA_ERR_UNSUPPORTED;
  for (int b = 0; b < B; ++b)
    if (valid_len[b] < 1 || valid_len[b] > n_k) return MHA_ERR_EMPTY_ROW;
  return MHA_OK;
}

// Key blocks of the attention kernels are 128 keys: with a padding mask the
// rows of K and V up to the valid length rounded up to a block are read (those
// past the length with weight exactly 0, so they must be finite), rows beyond
// are never read.
constexpr int KEY_BLOCK = 128;

// The three projections as one grouped GEMM: X_q (d_q wide) W_Q, X_k (d_k
// wide) W_K, X_v (d_v wide) W_V, each written head-split. With valid lengths
// (a padding mask) only the rows the attention step reads are computed: K and
// V rows below L_b rounded up to a key block, and the same Q rows when the
// query rows are positions of the same sequence (self_attention).
mha_status run_qkv(const void* X_q, const void* X_k, const void* X_v, const void* W_Q,
                   const void* W_K, const void* W_V, void* Q, void* K, void* V, int B, int n_q,
                   int n_k, int d_q, int d_k, int d_v, int h, int d_h, int d_vh,
                   const int32_t* valid_len, int self_attention, mha_dtype dt, int32_t* err,
                   cudaStream_t s) {
  GemmProblem p[3] = {
      head_split_problem(X_q, W_Q, Q, B, n_q, h, d_h, d_q),
      head_split_problem(X_k, W_K, K, B, n_k, h, d_h, d_k),
      head_split_problem(X_v, W_V, V, B, n_k, h, d_vh, d_v),
  };
  if (dt != MHA_DTYPE_BF16) return gemm_simt(p, 3, dt, s);
  if (!valid_len) return gemm_tc(p, 3, nullptr, err, s);
  int32_t need[MHA_MAX_PADDED_BATCH];
  for (int b = 0; b < B; ++b) {
    const long long r = ((long long)valid_len[b] + KEY_BLOCK - 1) / KEY_BLOCK * KEY_BLOCK;
    need[b] = (int32_t)(r < n_k ? r : n_k);
  }
  RowSelect sel{B, n_k, need, 0};
  p[0].select = self_attention ? 1 : 0;
  p[1].select = p[2].select = 1;
  return gemm_tc(p, 3, &sel, err, s);
}

// bf16 alignment the tensor-memory-access (TMA) GEMM needs: 16-byte row
// pitches and base addresses.
bool bf16_gemm_ok(int d_in, int width, const void* X, const void* W) {
  return d_in % 8 == 0 && width % 8 == 0 && aligned16(X) && aligned16(W);
}

mha_status run_attention(const AttnArgs& a, mha_dtype dt, cudaStream_t s) {
  if (dt == MHA_DTYPE_BF16 && tc_head_dims(a.d_h, a.d_vh)) return attention_tc(a, s);
  return attention_simt(a, dt, s);
}

// Y = Z W_O. With valid lengths (padded query rows of self-attention), the
// 128-row panels that hold only rows i >= L_b are written as zeros without a
// product (their Z rows are zeros); other rows are multiplied as usual.
mha_status run_out(const void* Z, const void* W_O, void* Y, int B, int n_q, int h, int d_vh,
                   int d_o, const int32_t* valid_len, mha_dtype dt, int32_t* err,
                   cudaStream_t s) {
  GemmProblem p = plain_problem(Z, W_O, Y, B * n_q, d_o, h * d_vh);
  if (dt != MHA_DTYPE_BF16) return gemm_simt(&p, 1, dt, s);
  if (!valid_len) return gemm_tc(&p, 1, nullptr, err, s);
  RowSelect sel{B, n_q, valid_len, 1};
  p.select = 1;
  return gemm_tc(&p, 1, &sel, err, s);
}

// Split over the keys of one attention call: 1 none, 0 automatic within the
// scratch, n > 1 n ranges; ws: device scratch (or null); zeroed: its counters
// were zeroed on the stream by the caller.
struct SplitReq {
  int nsplit;
  void* ws;
  size_t bytes;
  int zeroed;
};

// The attention step with its checks; head_gate (host, h floats) may be null.
mha_status attention_step(const void* Q, const void* K, const void* V, void* Z, int B, int n_q,
                          int n_k, int h, int d_h, int d_vh, float c, mha_mask_kind mask,
                          const int32_t* valid_len, int self_attention,
                          const float* head_gate, mha_dtype dt, int32_t* dev_error,
                          void* stream, SplitReq split = SplitReq{1, nullptr, 0, 0}) {
  if (!Q || !K || !V || !Z) return MHA_ERR_INVALID_ARG;
  if (B <= 0 || n_q <= 0 || n_k <= 0 || h <= 0 || d_h <= 0 || d_vh <= 0)
    return MHA_ERR_INVALID_ARG;
  if (!dtype_ok(dt) || !mask_ok(mask) || !isfinite(c)) return MHA_ERR_INVALID_ARG;
  if (has_causal(mask) && n_q != n_k) return MHA_ERR_INVALID_ARG;
  if (self_attention && n_q != n_k) return MHA_ERR_INVALID_ARG;
  mha_status st = check_valid_len(mask, valid_len, B, n_k);
  if (st != MHA_OK) return st;
  st = check_head_dims(d_h, d_vh, dt);
  if (st != MHA_OK) return st;
  if (!fits((long long)B * h, n_q, d_h) || !fits((long long)B * h, n_k, d_h) ||
      !fits((long long)B * h, n_k, d_vh) || !fits((long long)B * h, n_q, d_vh))
    return MHA_ERR_UNSUPPORTED;
  if (dt == MHA_DTYPE_BF16 && tc_head_dims(d_h, d_vh) &&
      (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(Z)))
    return MHA_ERR_UNSUPPORTED;
  AttnArgs a{};
  a.Q = Q;
  a.K = K;
  a.V = V;
  a.Z = Z;
  a.B = B;
  a.n_q = n_q;
  a.n_k = n_k;
  a.h = h;
  a.d_h = d_h;
  a.d_vh = d_vh;
  a.c = c;
  a.causal = has_causal(mask);
  a.padding = has_padding(mask);
  a.pad_queries = has_padding(mask) && self_attention;
  a.valid_len_host = valid_len;
  a.head_gate_host = head_gate;
  a.err = dev_error;
  a.nsplit = split.nsplit;
  a.split_ws = split.ws;
  a.split_ws_bytes = split.bytes;
  a.split_cnt_zeroed = split.zeroed;
  return run_attention(a, dt, static_cast<cudaStream_t>(stream));
}

}  // namespace

extern "C" {

size_t mha_workspace_size(int B, int n_q, int n_k, int d_model, int h, int d_h, int d_vh,
                          int d_o, mha_dtype dt) {
  if (B <= 0 || n_q <= 0 || n_k <= 0 || d_model <= 0 || h <= 0 || d_h <= 0 || d_vh <= 0 ||
      d_o <= 0 || !dtype_ok(dt))
    return 0;
  return layout(B, n_q, n_k, h, d_h, d_vh, dt).total;
}

mha_status mha_workspace_layout(int B, int n_q, int n_k, int h, int d_h, int d_vh,
                                mha_dtype dt, size_t offsets[6]) {
  if (!offsets || B <= 0 || n_q <= 0 || n_k <= 0 || h <= 0 || d_h <= 0 || d_vh <= 0 ||
      !dtype_ok(dt))
    return MHA_ERR_INVALID_ARG;
  const Layout L = layout(B, n_q, n_k, h, d_h, d_vh, dt);
  offsets[0] = 0;
  offsets[1] = L.q;
  offsets[2] = L.k;
  offsets[3] = L.v;
  offsets[4] = L.z;
  offsets[5] = L.total;
  return MHA_OK;
}

mha_status mha_qkv_projection(const void* X_q, const void* X_kv, const void* W_Q,
                              const void* W_K, const void* W_V, void* Q, void* K, void* V,
                              int B, int n_q, int n_k, int d_model, int h, int d_h, int d_vh,
                              mha_mask_kind mask, const int32_t* valid_len, mha_dtype dt,
                              int32_t* dev_error, void* stream) {
  if (!X_q || !W_Q || !W_K || !W_V || !Q || !K || !V) return MHA_ERR_INVALID_ARG;
  if (B <= 0 || n_q <= 0 || n_k <= 0 || d_model <= 0 || h <= 0 || d_h <= 0 || d_vh <= 0)
    return MHA_ERR_INVALID_ARG;
  if (!dtype_ok(dt) || !mask_ok(mask)) return MHA_ERR_INVALID_ARG;
  if (!X_kv && n_k != n_q) return MHA_ERR_INVALID_ARG;
  mha_status st = check_valid_len(mask, valid_len, B, n_k);
  if (st != MHA_OK) return st;
  st = check_head_dims(d_h, d_vh, dt);
  if (st != MHA_OK) return st;
  if (!fits(B, n_q, d_model) || !fits(B, n_k, d_model) || !fits(B, n_q, h * d_h) ||
      !fits(B, n_k, h * (long long)d_vh))
    return MHA_ERR_UNSUPPORTED;
  const void* Xk = X_kv ? X_kv : X_q;
  if (dt == MHA_DTYPE_BF16) {
    if (d_h % 8 || d_vh % 8 || !bf16_gemm_ok(d_model, h * d_h, X_q, W_Q) || !bf16_gemm_ok(d_model, h * d_h, Xk, W_K) ||
        !bf16_gemm_ok(d_model, h * d_vh, Xk, W_V) || !aligned16(Q) || !aligned16(K) ||
        !aligned16(V))
      return MHA_ERR_UNSUPPORTED;
  }
  return run_qkv(X_q, Xk, Xk, W_Q, W_K, W_V, Q, K, V, B, n_q, n_k, d_model, d_model, d_model, h,
                 d_h, d_vh, has_padding(mask) ? valid_len : nullptr, X_kv ? 0 : 1, dt, dev_error,
                 static_cast<cudaStream_t>(stream));
}

mha_status mha_attention(const void* Q, const void* K, const void* V, void* Z, int B, int n_q,
                         int n_k, int h, int d_h, int d_vh, float c, mha_mask_kind mask,
                         const int32_t* valid_len, int self_attention, mha_dtype dt,
                         int32_t* dev_error, void* stream) {
  return attention_step(Q, K, V, Z, B, n_q, n_k, h, d_h, d_vh, c, mask, valid_len,
                        self_attention, nullptr, dt, dev_error, stream);
}

size_t mha_attention_split_workspace_size(int B, int n_q, int n_k, int h, int d_h, int d_vh,
                                          int nsplit) {
  if (B <= 0 || n_q <= 0 || n_k <= 0 || h <= 0 || d_h <= 0 || d_vh <= 0 || nsplit < 0)
    return 0;
  if (!tc_head_dims(d_h, d_vh)) return 0;
  if (nsplit == 0) return attention_auto_split_bytes(B, n_q, n_k, h, d_vh);
  return attention_split_bytes(B, n_q, h, d_vh, attention_effective_splits(n_k, nsplit));
}

mha_status mha_attention_split(const void* Q, const void* K, const void* V, void* Z, int B,
                               int n_q, int n_k, int h, int d_h, int d_vh, float c,
                               mha_mask_kind mask, const int32_t* valid_len, int self_attention,
                               int nsplit, mha_dtype dt, void* workspace, size_t workspace_bytes,
                               int32_t* dev_error, void* stream) {
  if (nsplit < 0 || nsplit > MHA_MAX_KEY_SPLITS) return MHA_ERR_INVALID_ARG;
  if (workspace && (reinterpret_cast<uintptr_t>(workspace) & 255u)) return MHA_ERR_WORKSPACE;
  const bool tc = dt == MHA_DTYPE_BF16 && tc_head_dims(d_h, d_vh);
  if (nsplit > 1 && !tc) return MHA_ERR_UNSUPPORTED;
  if (nsplit > 1 && n_k > 0 && attention_effective_splits(n_k, nsplit) > 1 &&
      (!workspace || workspace_bytes < mha_attention_split_workspace_size(
                                           B, n_q, n_k, h, d_h, d_vh, nsplit)))
    return MHA_ERR_WORKSPACE;
  SplitReq split{nsplit, workspace, workspace ? workspace_bytes : 0, 0};
  return attention_step(Q, K, V, Z, B, n_q, n_k, h, d_h, d_vh, c, mask, valid_len,
                        self_attention, nullptr, dt, dev_error, stream, split);
}

mha_status mha_output_projection(const void* Z, const void* W_O, void* Y, int B, int n_q, int h,
                                 int d_vh, int d_o, const int32_t* valid_len, mha_dtype dt,
                                 int32_t* dev_error, void* stream) {
  if (!Z || !W_O || !Y) return MHA_ERR_INVALID_ARG;
  if (B <= 0 || n_q <= 0 || h <= 0 || d_vh <= 0 || d_o <= 0) return MHA_ERR_INVALID_ARG;
  if (!dtype_ok(dt)) return MHA_ERR_INVALID_ARG;
  if (valid_len) {
    const mha_status st = check_valid_len(MHA_MASK_PADDING, valid_len, B, n_q);
    if (st != MHA_OK) return st;
  }
  if (!fits(B, n_q, (long long)h * d_vh) || !fits(B, n_q, d_o)) return MHA_ERR_UNSUPPORTED;
  if (dt == MHA_DTYPE_BF16 &&
      ((h * d_vh) % 8 || d_o % 8 || !aligned16(Z) || !aligned16(W_O) || !aligned16(Y)))
    return MHA_ERR_UNSUPPORTED;
  return run_out(Z, W_O, Y, B, n_q, h, d_vh, d_o, valid_len, dt, dev_error,
                 static_cast<cudaStream_t>(stream));
}

mha_status mha_forward_general(const void* X_q, const void* X_k, const void* X_v,
                               const void* W_Q, const void* W_K, const void* W_V,
                               const void* W_O, void* Y, int B, int n_q, int n_k, int d_q,
                               int d_k, int d_v, int h, int d_h, int d_vh, int d_o, float c,
                               mha_mask_kind mask, const int32_t* valid_len, int self_attention,
                               const float* head_gate, mha_dtype dt, void* workspace,
                               size_t workspace_bytes, void* stream) {
  // Host-side checks, all before anything is enqueued.
  if (!X_q || !X_k || !X_v || !W_Q || !W_K || !W_V || !W_O || !Y) return MHA_ERR_INVALID_ARG;
  if (B <= 0 || n_q <= 0 || n_k <= 0 || d_q <= 0 || d_k <= 0 || d_v <= 0 || h <= 0 ||
      d_h <= 0 || d_vh <= 0 || d_o <= 0)
    return MHA_ERR_INVALID_ARG;
  if (!dtype_ok(dt) || !mask_ok(mask) || !isfinite(c)) return MHA_ERR_INVALID_ARG;
  if (self_attention && n_k != n_q) return MHA_ERR_INVALID_ARG;
  if (has_causal(mask) && n_q != n_k) return MHA_ERR_INVALID_ARG;
  mha_status st = check_valid_len(mask, valid_len, B, n_k);
  if (st != MHA_OK) return st;
  st = check_head_dims(d_h, d_vh, dt);
  if (st != MHA_OK) return st;
  if (head_gate) {
    if (h > MHA_MAX_GATED_HEADS) return MHA_ERR_UNSUPPORTED;
    for (int i = 0; i < h; ++i)
      if (!isfinite(head_gate[i])) return MHA_ERR_INVALID_ARG;
  }
  if (!fits(B, n_q, d_q) || !fits(B, n_k, d_k) || !fits(B, n_k, d_v) ||
      !fits(B, n_q, (long long)h * d_h) || !fits(B, n_k, (long long)h * d_h) ||
      !fits(B, n_k, (long long)h * d_vh) || !fits(B, n_q, d_o))
    return MHA_ERR_UNSUPPORTED;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return MHA_ERR_WORKSPACE;
  const Layout L = layout(B, n_q, n_k, h, d_h, d_vh, dt);
  if (workspace_bytes < L.total) return MHA_ERR_WORKSPACE;
  if (dt == MHA_DTYPE_BF16 &&
      (d_h % 8 || d_vh % 8 || !bf16_gemm_ok(d_q, h * d_h, X_q, W_Q) ||
       !bf16_gemm_ok(d_k, h * d_h, X_k, W_K) ||
       !bf16_gemm_ok(d_v, h * d_vh, X_v, W_V) || !bf16_gemm_ok(h * d_vh, d_o, W_O, Y)))
    return MHA_ERR_UNSUPPORTED;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  int32_t* err = reinterpret_cast<int32_t*>(ws);
  void* Q = ws + L.q;
  void* K = ws + L.k;
  void* V = ws + L.v;
  void* Z = ws + L.z;
  if (cudaMemsetAsync(err, 0, sizeof(int32_t), s) != cudaSuccess) return MHA_ERR_CUDA;
  // the split counters are zeroed here, ahead of the projection, so that the
  // attention kernel still follows the projection kernel directly
  SplitReq split{0, nullptr, 0, 1};
  if (L.split_bytes > 0) {
    split.ws = ws + L.split;
    split.bytes = L.split_bytes;
    if (cudaMemsetAsync(split.ws, 0, attention_split_counter_bytes(B, n_q, h), s) != cudaSuccess)
      return MHA_ERR_CUDA;
  }
  const int32_t* lens = has_padding(mask) ? valid_len : nullptr;
  st = run_qkv(X_q, X_k, X_v, W_Q, W_K, W_V, Q, K, V, B, n_q, n_k, d_q, d_k, d_v, h, d_h, d_vh,
               lens, self_attention ? 1 : 0, dt, err, s);
  if (st != MHA_OK) return st;
  st = attention_step(Q, K, V, Z, B, n_q, n_k, h, d_h, d_vh, c, mask, valid_len,
                      self_attention ? 1 : 0, head_gate, dt, err, stream, split);
  if (st != MHA_OK) return st;
  // padded query rows (self-attention) are zeros in Z, so in Y
  return mha_output_projection(Z, W_O, Y, B, n_q, h, d_vh, d_o, self_attention ? lens : nullptr,
                               dt, err, stream);
}

mha_status mha_forward(const void* X_q, const void* X_kv, const void* W_Q, const void* W_K,
                       const void* W_V, const void* W_O, void* Y, int B, int n_q, int n_k,
                       int d_model, int h, int d_h, int d_vh, int d_o, float c,
                       mha_mask_kind mask, const int32_t* valid_len, mha_dtype dt,
                       void* workspace, size_t workspace_bytes, void* stream) {
  if (!X_q) return MHA_ERR_INVALID_ARG;
  const bool self_attn = X_kv == nullptr;
  if (self_attn && n_k != n_q) return MHA_ERR_INVALID_ARG;
  const void* Xkv = self_attn ? X_q : X_kv;
  return mha_forward_general(X_q, Xkv, Xkv, W_Q, W_K, W_V, W_O, Y, B, n_q, n_k, d_model,
                             d_model, d_model, h, d_h, d_vh, d_o, c, mask, valid_len,
                             self_attn ? 1 : 0, nullptr, dt, workspace, workspace_bytes,
                             stream);
}

size_t mha_decode_workspace_size(int B, int n_q, int n_k, int h, int d_vh) {
  if (B <= 0 || n_q <= 0 || n_k <= 0 || h <= 0 || d_vh <= 0) return 0;
  return decode_workspace_bytes(B, n_q, n_k, h, d_vh);
}

mha_status mha_attention_decode(const void* Q, const void* K, const void* V, void* Z, int B,
                                int n_q, int n_k, int h, int d_h, int d_vh, float c,
                                const int32_t* cache_len, int causal_tail, mha_dtype dt,
                                void* workspace, size_t workspace_bytes, void* stream) {
  if (!Q || !K || !V || !Z) return MHA_ERR_INVALID_ARG;
  if (B <= 0 || n_q <= 0 || n_k <= 0 || h <= 0 || d_h <= 0 || d_vh <= 0)
    return MHA_ERR_INVALID_ARG;
  if (!dtype_ok(dt) || !isfinite(c)) return MHA_ERR_INVALID_ARG;
  // the kernels take the cache lengths as a fixed-size launch argument
  if (B > MHA_MAX_PADDED_BATCH) return MHA_ERR_UNSUPPORTED;
  if (cache_len) {
    for (int b = 0; b < B; ++b)
      if (cache_len[b] < 1 || cache_len[b] > n_k || (causal_tail && cache_len[b] < n_q))
        return MHA_ERR_EMPTY_ROW;
  } else if (causal_tail && n_k < n_q) {
    return MHA_ERR_EMPTY_ROW;
  }
  if (d_h > MAX_HEAD_DIM || d_vh > MAX_HEAD_DIM || n_k > 65536) return MHA_ERR_UNSUPPORTED;
  if (!fits((long long)B * h, n_q, d_h) || !fits((long long)B * h, n_k, d_h) ||
      !fits((long long)B * h, n_k, d_vh) || !fits((long long)B * h, n_q, d_vh))
    return MHA_ERR_UNSUPPORTED;
  if (dt == MHA_DTYPE_BF16 &&
      (d_h % 8 || !aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(Z)))
    return MHA_ERR_UNSUPPORTED;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 15u) ||
      workspace_bytes < decode_workspace_bytes(B, n_q, n_k, h, d_vh))
    return MHA_ERR_WORKSPACE;
  DecodeArgs a{};
  a.Q = Q;
  a.K = K;
  a.V = V;
  a.Z = Z;
  a.part = workspace;
  a.B = B;
  a.n_q = n_q;
  a.n_k = n_k;
  a.h = h;
  a.d_h = d_h;
  a.d_vh = d_vh;
  a.c = c;
  a.causal_tail = causal_tail ? 1 : 0;
  a.cache_len_host = cache_len;
  return attention_decode(a, dt, static_cast<cudaStream_t>(stream));
}

mha_status mha_get_device_error(void* error_word, void* stream) {
  if (!error_word) return MHA_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t v = 0;
  if (cudaMemcpyAsync(&v, error_word, sizeof(v), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return MHA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MHA_ERR_CUDA;
  if (v != 0 && cudaMemsetAsync(error_word, 0, sizeof(int32_t), s) != cudaSuccess)
    return MHA_ERR_CUDA;
  return static_cast<mha_status>(v);
}

const char* mha_status_string(mha_status s) {
  switch (s) {
    case MHA_OK: return "ok";
    case MHA_ERR_INVALID_ARG: return "invalid argument";
    case MHA_ERR_UNSUPPORTED: return "unsupported shape, alignment or size";
    case MHA_ERR_EMPTY_ROW: return "a query row has no allowed key (valid length outside [1, n_k])";
    case MHA_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case MHA_ERR_CUDA: return "CUDA runtime or launch error";
    case MHA_ERR_DEVICE_TIMEOUT: return "a kernel gave up waiting on one of its barriers";
  }
  return "unknown status";
}

mha_status mha_selftest_wait_timeout(int32_t* dev_error, uint64_t limit_ns, void* stream) {
  if (!dev_error) return MHA_ERR_INVALID_ARG;
  if (limit_ns < 1000ull) limit_ns = 1000ull;
  if (limit_ns > 10000000000ull) limit_ns = 10000000000ull;
  return selftest_wait(dev_error, limit_ns, static_cast<cudaStream_t>(stream));
}

mha_status mha_attention_plan(int B, int n_q, int n_k, int h, int d_h, int d_vh,
                              mha_mask_kind mask, const int32_t* valid_len, int self_attention,
                              int nsplit, int num_sms, int32_t* grid, int32_t* records,
                              size_t max_records, size_t* n_records) {
  if (!grid || !n_records || num_sms < 1) return MHA_ERR_INVALID_ARG;
  if (nsplit < 0 || nsplit > MHA_MAX_KEY_SPLITS) return MHA_ERR_INVALID_ARG;
  if (B <= 0 || n_q <= 0 || n_k <= 0 || h <= 0 || d_h <= 0 || d_vh <= 0)
    return MHA_ERR_INVALID_ARG;
  if (!mask_ok(mask)) return MHA_ERR_INVALID_ARG;
  if (has_causal(mask) && n_q != n_k) return MHA_ERR_INVALID_ARG;
  if (self_attention && n_q != n_k) return MHA_ERR_INVALID_ARG;
  const mha_status st = check_valid_len(mask, valid_len, B, n_k);
  if (st != MHA_OK) return st;
  if (!tc_head_dims(d_h, d_vh)) return MHA_ERR_UNSUPPORTED;
  AttnArgs a{};
  a.B = B;
  a.n_q = n_q;
  a.n_k = n_k;
  a.h = h;
  a.d_h = d_h;
  a.d_vh = d_vh;
  a.causal = has_causal(mask);
  a.padding = has_padding(mask);
  a.pad_queries = has_padding(mask) && self_attention;
  a.valid_len_host = valid_len;
  // the plan launches nothing: the scratch is only sized, never touched
  static char no_scratch;
  a.nsplit = nsplit;
  a.split_ws_bytes = mha_attention_split_workspace_size(B, n_q, n_k, h, d_h, d_vh, nsplit);
  a.split_ws = a.split_ws_bytes > 0 ? &no_scratch : nullptr;
  int g = 0;
  const mha_status ps = attention_tc_plan(a, num_sms, &g, records, max_records, n_records);
  *grid = g;
  return ps;
}

uint64_t mha_kernel_launch_count(void) { return g_launches.load(); }

const char* mha_version(void) { return "head_scaled_dot_gb300 0.1 (sm_103a)"; }

}  // extern "C"
