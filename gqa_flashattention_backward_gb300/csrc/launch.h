// Internal launcher declarations shared by the translation units of the CUDA path.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include "common.cuh"

namespace gqa {

// Tensor maps of one call (built on the host, passed by value to kernels).
struct Maps {
  CUtensorMap q, k, v, o, dout;  // 16-bit tensors as 4-D (D, S, H, B) with the caller's strides,
                                 // 128B swizzle, box 64 columns x rows of one (b, h)
  CUtensorMap dq_acc;            // fp32 [B*Hq][S][Dqk], box 32 x 32, 128B swizzle (bulk reduce)
  CUtensorMap dk_acc, dv_acc;    // fp32 [B*Hkv][S][D]
};

enum DqMode : int { kDqNone = 0, kDqRedV4 = 1, kDqBulk = 2, kDqScalar = 3, kDqStore = 4 };

struct KvLaunch {
  int group_tmem;     // 1: dK/dV summed over the group in TMEM; 0: per-head CTA + atomics
  int dq_mode;        // DqMode; kDqNone when dQ comes from the query-stationary pass
  int kv_red_mode;    // DqMode values reused for the dK/dV atomics of group_tmem == 0
  void* dk;           // outputs (group_tmem)
  void* dv;
};

cudaError_t launch_preprocess(const Problem& p, int dtype_bf16, const void* o, const void* dout, const float* lse,
                              float* delta, bool zero_dq, int num_sms, cudaStream_t st);
cudaError_t launch_cast(const float* acc, void* out, int B, int H, int S, int D, const Strides& st, float mul,
                        int dtype_bf16, int num_sms, cudaStream_t st_);
cudaError_t launch_dsink(int B, int Hq, int S, const float* sink, const float* lse, const float* delta,
                         float* dsink, cudaStream_t st);
cudaError_t launch_selftest_wait(int* err, long long limit, cudaStream_t st);

// One-pass forward (O, LSE); the K / V tensor-map box height (keys per tile) it needs.
cudaError_t launch_fwd(const Problem& p, int dtype_bf16, const Maps& m, const float* sink, void* o, float* lse,
                       cudaStream_t st);
int fwd_kernel_bk(int Dqk);
// Query-stationary dQ pass (deterministic mode, head dim 192); keys per tile of it.
cudaError_t launch_dq(const Problem& p, int dtype_bf16, const Maps& m, void* dq, cudaStream_t st);
int q_kernel_bk();

// Key/value-stationary backward main kernel.
cudaError_t launch_bwd_kv(const Problem& p, int dtype_bf16, const Maps& m, const KvLaunch& kl, cudaStream_t st);

}  // namespace gqa
