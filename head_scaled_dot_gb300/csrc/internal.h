// internal.h - host-side interfaces shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "mha.h"

namespace mha {

// One GEMM of a grouped launch: out = A (M x K, row-major) * W (K x N,
// row-major), written through the index map
//   dest(m, n) = (m / rows_per_group) * s_group_row + (n / cols_per_group) * s_group_col
//              + (m % rows_per_group) * s_row + (n % cols_per_group)
// which covers both the plain row-major output (rows_per_group = M,
// cols_per_group = N, s_row = N) and the head split (B,T,h*d) -> (B,h,T,d)
// (rows_per_group = T, cols_per_group = d, s_group_row = h*T*d,
// s_group_col = T*d, s_row = d).
struct GemmProblem {
  const void* A;
  const void* W;
  void* out;
  int M, N, K;
  int rows_per_group, cols_per_group;
  long long s_group_row, s_group_col, s_row;
  int select;  // rows chosen by the launch's RowSelect (else every row)
};

static inline GemmProblem plain_problem(const void* A, const void* W, void* out, int M, int N,
                                        int K) {
  GemmProblem p{A, W, out, M, N, K, M, N, 0, 0, (long long)N, 0};
  return p;
}

static inline GemmProblem head_split_problem(const void* A, const void* W, void* out, int B,
                                             int T, int h, int d, int K) {
  GemmProblem p{A,  W, out, B * T, h * d, K, T, d, (long long)h * T * d, (long long)T * d,
                (long long)d, 0};
  return p;
}

// The rows of a grouped GEMM that matter, for the problems with `select`
// set: their A rows are B blocks of rows_per_batch rows (one block per batch
// item), and in block b only the first need[b] rows matter (1 <= need[b] <=
// rows_per_batch). 128-row output tiles without such a row are not
// multiplied: they are skipped (their output rows are left as they were), or,
// with zero_rest (one problem only), written as zeros.
struct RowSelect {
  int B;
  int rows_per_batch;
  const int32_t* need;  // host, B entries
  int zero_rest;
};

// Attention step arguments (Q, K, V head-split; Z concatenated).
struct AttnArgs {
  const void* Q;
  const void* K;
  const void* V;
  void* Z;
  int B, n_q, n_k, h, d_h, d_vh;
  float c;
  int causal;           // keys j <= i only
  int padding;          // keys j < valid_len[b]
  int pad_queries;      // rows i >= valid_len[b] are not computed (Z row = 0)
  const int32_t* valid_len_host;  // B entries when padding
  const float* head_gate_host;    // h entries, or null (all 1): head i's output is scaled by it
  int32_t* err;
  // Split over the keys (tensor-core path): 1 none, 0 automatic (within
  // split_ws_bytes), n > 1 that many key ranges (fewer when n_k has fewer
  // 128-key blocks). split_ws: device scratch for the ranges' summaries
  // (attention_split_bytes), 256-byte aligned, or null; split_cnt_zeroed: the
  // caller zeroed its first split_counter bytes on the call's stream.
  int nsplit;
  void* split_ws;
  size_t split_ws_bytes;
  int split_cnt_zeroed;
};

// Attention of a few query rows over a key/value cache, split over the keys
// (decode.cu). Q (B,h,n_q,d_h), K (B,h,n_k,d_h), V (B,h,n_k,d_vh) head-split;
// Z (B,n_q,h*d_vh); part: decode_workspace_bytes of device scratch.
struct DecodeArgs {
  const void* Q;
  const void* K;
  const void* V;
  void* Z;
  void* part;
  int B, n_q, n_k, h, d_h, d_vh;
  float c;
  int causal_tail;                 // row i sees keys j <= L_b - n_q + i
  const int32_t* cache_len_host;   // B entries, or null (every length n_k)
};

size_t decode_workspace_bytes(int B, int n_q, int n_k, int h, int d_vh);
mha_status attention_decode(const DecodeArgs& a, mha_dtype dt, cudaStream_t s);

// Raises the dynamic shared-memory limit of `kernel` to `bytes` on the
// current device, once per (device, kernel): the attribute belongs to the
// device, not to the process. Thread-safe; false on a CUDA error.
bool ensure_smem_limit(const void* kernel, int bytes);
// CTAs of `kernel` that fit on one SM of the current device at once (at
// least 1), asked once per (device, kernel). Thread-safe.
int resident_ctas(const void* kernel, int threads, int smem_bytes);

// Kernel limit for bounded waits (nanoseconds).
uint64_t wait_limit_ns();
void count_launch(int n = 1);
int num_sms();

// CUDA-core kernels (fp32; the bf16 instantiation is kept for tests).
mha_status gemm_simt(const GemmProblem* probs, int nprob, mha_dtype dt, cudaStream_t s);
mha_status attention_simt(const AttnArgs& a, mha_dtype dt, cudaStream_t s);

// Tensor-core kernels (bf16).
// Problems with the same A (pointer, M and K) and the same `select` that are
// next to each other in probs form a group: its tiles run M panel by M panel,
// each panel through every problem of the group, so the panel of A is read
// from memory once. sel may be null (every row).
mha_status gemm_tc(const GemmProblem* probs, int nprob, const RowSelect* sel, int32_t* err,
                   cudaStream_t s);
mha_status attention_tc(const AttnArgs& a, cudaStream_t s);
// Scratch of a split over the keys into nsplit ranges (0 for nsplit < 2):
// per-tile counters, then one summary slot per (tile pair, tile, range).
size_t attention_split_bytes(int B, int n_q, int h, int d_vh, int nsplit);
// Scratch the automatic split may use for these sizes (0: it never splits).
size_t attention_auto_split_bytes(int B, int n_q, int n_k, int h, int d_vh);
// Leading bytes of the split scratch that hold the counters (zeroed per call).
size_t attention_split_counter_bytes(int B, int n_q, int h);
// Key ranges a requested split of n_k keys into nsplit ranges gives (1: none).
int attention_effective_splits(int n_k, int nsplit);
// The schedule attention_tc would launch on a GPU with num_sms SMs: the grid
// size and, CTA by CTA in processing order, one record {cta, b, head, q0,
// ntiles, key0, key1} per unit (query rows [q0, q0 + 128 ntiles) of one head
// over keys [key0, key1)), at most max_records of them written; *n_records =
// all units. Host only.
mha_status attention_tc_plan(const AttnArgs& a, int num_sms, int* grid, int32_t* records,
                             size_t max_records, size_t* n_records);

// TMA descriptors (cuTensorMapEncodeTiled through the runtime's driver entry
// point). dims/strides innermost first; strides in bytes for dims 1..rank-1.
bool make_tmap_bf16(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                    const uint64_t* strides_bytes, const uint32_t* box, bool swizzle128);

mha_status selftest_wait(int32_t* err, uint64_t limit_ns, cudaStream_t s);

// Launches kernel(arg) with programmatic stream serialization: it may begin
// launching while the previous kernel of the stream is still running, and
// must call grid_dep_wait before it reads or writes global memory.
template <typename Arg>
cudaError_t launch_dependent(void (*kernel)(Arg), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t s, const Arg& arg) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, arg);
}

}  // namespace mha
