// Memory-bound kernels of the backward path:
//   preprocess  : Delta_i = sum_d dO_id * O_id; tiled row statistics for the
//                 main kernels; zero the fp32 accumulators.
//                 (tilelang-ascend PR #1638 "Add GQA Sink Backward BHSD": the
//                 9->6 commit's preprocess kernel; Phase0(Delta) = sum(O*dO).)
//   postprocess : fp32 accumulators -> fp16/bf16 outputs (dual-output cast of the
//                 same PR's 9->6 commit; the 4->2 commit's "fp32 atomic_add
//                 then cast").
//   dsink       : dsink_h = -sum_{b,i} exp(sink_h - lse) * Delta ("Kernel 9: Dsink"), one
//                 eight-CTA cluster per head.
// All are grid-stride kernels sized to a multiple of the SM count with 16-byte
// vector accesses.
#include <cooperative_groups.h>
#include <type_traits>
#include "common.cuh"
#include "umma.cuh"
#include "launch.h"

namespace gqa {

template <typename T>
__device__ __forceinline__ float2 to_f2(uint32_t u);
template <>
__device__ __forceinline__ float2 to_f2<__half>(uint32_t u) {
  return __half22float2(*reinterpret_cast<__half2*>(&u));
}
template <>
__device__ __forceinline__ float2 to_f2<__nv_bfloat16>(uint32_t u) {
  return __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&u));
}

// Locate sequence s and local index of token `row` on the S axis (packed case).
__device__ __forceinline__ int find_seq(const int32_t* cu, int nseqs, int row) {
  int lo = 0, hi = nseqs - 1;  // largest s with cu[s] <= row, among non-empty candidates
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(cu + mid) <= row) lo = mid;
    else hi = mid - 1;
  }
  // skip empty sequences that share the same start
  while (lo + 1 < nseqs && __ldg(cu + lo + 1) <= row) ++lo;
  return lo;
}

// One query row of an xfold tile: 16 bf16 values in the no-swizzle K-major core-matrix layout
// (8 rows x 16 bytes per core matrix; the 8-row groups 256 bytes apart, the two K halves
// 128 bytes apart).  K columns 0-2 hold -LSE/scale as three bf16 terms hi + mid + lo, which add up
// to the fp32 value exactly (each step's remainder has at most 16, then 8 significant bits) and
// keep fp32's range; columns 8-10 hold -Delta the same way; the rest are zero.  Adding this row
// through one K=16 MMA against a ones operand subtracts LSE/scale from every logit of the row
// (resp. Delta from every dP) in fp32.
__device__ __forceinline__ uint2 split3(float x) {
  x = fminf(fmaxf(x, -1e30f), 1e30f);  // -inf (padding rows) -> a value that zeroes exp2
  const __nv_bfloat16 hi = __float2bfloat16_rn(x);
  const float r = x - __bfloat162float(hi);
  const __nv_bfloat16 mid = __float2bfloat16_rn(r);
  const __nv_bfloat16 lo = __float2bfloat16_rn(r - __bfloat162float(mid));
  return make_uint2(static_cast<uint32_t>(__bfloat16_as_ushort(hi)) | (static_cast<uint32_t>(__bfloat16_as_ushort(mid)) << 16),
                    static_cast<uint32_t>(__bfloat16_as_ushort(lo)));
}
__device__ __forceinline__ void write_fold_row(uint8_t* tile, int q, float xl, float xd) {
  uint8_t* row = tile + (q >> 3) * 256 + (q & 7) * 16;
  const uint2 l = split3(xl), d = split3(xd);
  *reinterpret_cast<uint4*>(row) = make_uint4(l.x, l.y, 0u, 0u);
  *reinterpret_cast<uint4*>(row + 128) = make_uint4(d.x, d.y, 0u, 0u);
}

// The main kernel's sequence order (sched_fill), by one block from the packed key lengths.  A
// malformed or over-long sequence counts 0 tiles (the main kernel reports it and skips it).
__device__ void build_schedule(const Problem& p) {
  __shared__ int key[kSchedMaxSeqs];
  const int n = p.nseqs;
  const int32_t* cu = p.cu_seqlens_k ? p.cu_seqlens_k : p.cu_seqlens;
  for (int q = threadIdx.x; q < n; q += blockDim.x) {
    const int a = __ldg(cu + q), e = __ldg(cu + q + 1);
    const int len = e - a;
    key[q] = (len < 0 || a < 0 || e > p.Sk || len > p.max_len_k) ? 0 : (len + 127) / 128;
  }
  __syncthreads();
  sched_fill(p.sched, key, n, threadIdx.x, blockDim.x);
}

// 8 threads per row; each thread covers Dv/8 elements.
template <typename T, int DV>
__global__ void __launch_bounds__(256) preprocess_kernel(Problem p, const T* __restrict__ o,
                                                         const T* __restrict__ dout, const float* __restrict__ lse,
                                                         float* __restrict__ delta, int zero_dq) {
  constexpr int PER = DV / 8;        // elements per thread
  constexpr int VEC = PER / 8;       // uint4 loads per thread per tensor
  const long long nrows = static_cast<long long>(p.B) * p.Hq * p.S;
  if (p.sched && blockIdx.x == 0) build_schedule(p);
  const int sub = threadIdx.x & 7;
  const long long stride = static_cast<long long>(gridDim.x) * (blockDim.x >> 3);
  for (long long r = static_cast<long long>(blockIdx.x) * (blockDim.x >> 3) + (threadIdx.x >> 3); r < nrows;
       r += stride) {
    const int i = static_cast<int>(r % p.S);
    const int h = static_cast<int>((r / p.S) % p.Hq);
    const int b = static_cast<int>(r / (static_cast<long long>(p.S) * p.Hq));
    const uint4* po = reinterpret_cast<const uint4*>(o + p.o_st.row(b, h, i) + sub * PER);
    const uint4* pd = reinterpret_cast<const uint4*>(dout + p.do_st.row(b, h, i) + sub * PER);
    float acc = 0.f;
#pragma unroll
    for (int v = 0; v < VEC; ++v) {
      const uint4 a = __ldg(po + v), b = __ldg(pd + v);
      const uint32_t aa[4] = {a.x, a.y, a.z, a.w}, bb[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 x = to_f2<T>(aa[e]), y = to_f2<T>(bb[e]);
        acc = fmaf(x.x, y.x, acc);
        acc = fmaf(x.y, y.y, acc);
      }
    }
    // the row's eight threads are one aligned group of eight lanes, all active together (a warp's other
    // rows may have left the loop at the end of the rows): the mask names exactly that group
    const unsigned grp = 0xFFu << (threadIdx.x & 24);
    acc += __shfl_xor_sync(grp, acc, 1);
    acc += __shfl_xor_sync(grp, acc, 2);
    acc += __shfl_xor_sync(grp, acc, 4);
    int s, il, len;
    if (p.cu_seqlens) {
      s = find_seq(p.cu_seqlens, p.nseqs, i);
      const int st = __ldg(p.cu_seqlens + s);
      il = i - st;
      len = __ldg(p.cu_seqlens + s + 1) - st;
    } else {
      s = b;
      il = i;
      len = p.S;
    }
    const bool ok = len <= p.max_len;
    if (sub == 0) {
      delta[r] = acc;
      if (ok) {
        const size_t base = stat_index(p, h, s, il / kStatTile) + (il % kStatTile);
        p.nlse2[base] = -__ldg(lse + r) * kLog2e;
        p.ndelta[base] = -acc;
        if (p.xfold)
          write_fold_row(p.xfold + stat_index(p, h, s, il / kStatTile) * kFoldRowBytes, il % kStatTile,
                         -__ldg(lse + r) / p.scale, -acc);
      } else if (il == 0) {
        atomicCAS(p.err, 0, kErrSeqTooLong);
      }
    }
    // the last row of a sequence fills the padding rows of its final stat tile
    if (ok && il == len - 1 && (len % kStatTile) != 0) {
      const size_t base = stat_index(p, h, s, il / kStatTile);
      for (int pr = (len % kStatTile) + sub; pr < kStatTile; pr += 8) {
        p.nlse2[base + pr] = __int_as_float(0xff800000);  // -inf: exp2(x - inf) = 0
        p.ndelta[base + pr] = 0.f;
        if (p.xfold) write_fold_row(p.xfold + base * kFoldRowBytes, pr, -INFINITY, 0.f);
      }
    }
    if (zero_dq) {
      float4* z = reinterpret_cast<float4*>(p.dq_acc + r * p.Dqk);
      for (int c = sub; c < p.Dqk / 4; c += 8) z[c] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
}

// out row (b, h, s) = dtype(acc row * mul): acc is contiguous fp32 [B, H, S, D], out has the caller's
// layout; 8 elements (two 16-byte loads, one 16-byte store) per thread-iteration.  Grid y walks the
// (b, h) pairs and x the S * D / 8 chunks of one pair, so a chunk's row comes from one division by a
// compile-time constant (64-bit divisions by S and H per chunk kept the kernel instruction-bound).
template <typename T, int D>
__global__ void __launch_bounds__(256) cast_kernel(const float* __restrict__ acc, T* __restrict__ out, int H, int S,
                                                   int BH, Strides st, float mul) {
  constexpr int PER_ROW = D / 8;
  constexpr bool BF = std::is_same<T, __nv_bfloat16>::value;
  const int n = S * PER_ROW;  // chunks of one (b, h)
  for (int bh = blockIdx.y; bh < BH; bh += gridDim.y) {
    const int b = bh / H, h = bh - b * H;
    const float4* a4 = reinterpret_cast<const float4*>(acc + static_cast<size_t>(bh) * S * D);
    for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < n; e += gridDim.x * blockDim.x) {
      const int si = e / PER_ROW, c8 = e - si * PER_ROW;
      const float4 a = __ldg(a4 + 2 * static_cast<size_t>(e));
      const float4 c = __ldg(a4 + 2 * static_cast<size_t>(e) + 1);
      uint4 r;
      r.x = pack2<BF>(a.x * mul, a.y * mul);
      r.y = pack2<BF>(a.z * mul, a.w * mul);
      r.z = pack2<BF>(c.x * mul, c.y * mul);
      r.w = pack2<BF>(c.z * mul, c.w * mul);
      *reinterpret_cast<uint4*>(out + st.row(b, h, si) + 8 * c8) = r;
    }
  }
}

// One cluster of kDsinkCluster CTAs per head: CTA c of the cluster sums every kDsinkCluster-th block
// of the head's B*S rows in a fixed order, then rank 0 adds the CTAs' sums in rank order through
// distributed shared memory -- deterministic, and eight CTAs per head stream LSE / Delta instead of one.
constexpr int kDsinkCluster = 8;
constexpr int kDsinkThreads = 256;

__global__ void __cluster_dims__(kDsinkCluster, 1, 1) __launch_bounds__(kDsinkThreads)
    dsink_kernel(int B, int Hq, int S, const float* __restrict__ sink, const float* __restrict__ lse,
                 const float* __restrict__ delta, float* __restrict__ dsink) {
  namespace cg = cooperative_groups;
  cg::cluster_group cl = cg::this_cluster();
  const int h = blockIdx.x / kDsinkCluster;
  const int c = static_cast<int>(cl.block_rank());
  const float sh = __ldg(sink + h);
  const long long n = static_cast<long long>(B) * S;  // this head's rows over the batch
  float acc = 0.f;
  for (long long e = static_cast<long long>(c) * kDsinkThreads + threadIdx.x; e < n;
       e += static_cast<long long>(kDsinkCluster) * kDsinkThreads) {
    const long long b = e / S, i = e - b * S;
    const size_t r = (static_cast<size_t>(b) * Hq + h) * S + i;
    acc += __expf(sh - __ldg(lse + r)) * __ldg(delta + r);
  }
  __shared__ float red[kDsinkThreads / 32];
  __shared__ float part;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    float v = 0.f;
    for (int wi = 0; wi < kDsinkThreads / 32; ++wi) v += red[wi];
    part = v;
  }
  cl.sync();  // every CTA's sum is in its shared memory
  if (c == 0 && threadIdx.x == 0) {
    float tot = 0.f;
    for (int k = 0; k < kDsinkCluster; ++k) tot += *cl.map_shared_rank(&part, k);
    dsink[h] = -tot;
  }
  cl.sync();  // the peers keep their shared memory until rank 0 has read it
}

// Waits on a barrier that nothing completes: exercises the timeout path.
__global__ void selftest_wait_kernel(int* err, long long limit) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  WaitGuard g{err, &abort_flag, limit};
  if (threadIdx.x == 0) mbar_wait(&bar, 0, g, 0x7e);
  __syncthreads();
}

// ---------------------------------------------------------------- launchers
cudaError_t launch_preprocess(const Problem& p, int dtype_bf16, const void* o, const void* dout, const float* lse,
                              float* delta, bool zero_dq, int num_sms, cudaStream_t st) {
  const long long rows = static_cast<long long>(p.B) * p.Hq * p.S;
  long long blocks = (rows + 31) / 32;
  const long long cap = static_cast<long long>(num_sms) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
#define GQA_PRE(T, DV)                                                                                \
  preprocess_kernel<T, DV><<<static_cast<unsigned>(blocks), 256, 0, st>>>(                            \
      p, static_cast<const T*>(o), static_cast<const T*>(dout), lse, delta, zero_dq)
  if (dtype_bf16) {
    if (p.Dv == 64) GQA_PRE(__nv_bfloat16, 64);
    else GQA_PRE(__nv_bfloat16, 128);
  } else {
    if (p.Dv == 64) GQA_PRE(__half, 64);
    else GQA_PRE(__half, 128);
  }
#undef GQA_PRE
  return cudaGetLastError();
}

cudaError_t launch_cast(const float* acc, void* out, int B, int H, int S, int D, const Strides& st, float mul,
                        int dtype_bf16, int num_sms, cudaStream_t st_) {
  const long long bh = static_cast<long long>(B) * H;
  if (bh <= 0 || S <= 0) return cudaSuccess;
  if (static_cast<long long>(S) * (D / 8) > 0x7fffffffLL || bh > 0x7fffffffLL) return cudaErrorInvalidValue;
  // about eight 256-thread blocks per SM in all, spread over the (b, h) pairs
  const long long per_bh = (static_cast<long long>(S) * (D / 8) + 255) / 256;
  const unsigned gy = static_cast<unsigned>(bh < 65535 ? bh : 65535);
  long long gx = (static_cast<long long>(num_sms) * 8 + gy - 1) / gy;
  if (gx > per_bh) gx = per_bh;
  if (gx < 1) gx = 1;
  const dim3 grid(static_cast<unsigned>(gx), gy);
#define GQA_CAST(T, DD)                                                                                 \
  cast_kernel<T, DD><<<grid, 256, 0, st_>>>(acc, static_cast<T*>(out), H, S, static_cast<int>(bh), st, mul)
  if (dtype_bf16) {
    if (D == 64) GQA_CAST(__nv_bfloat16, 64);
    else if (D == 128) GQA_CAST(__nv_bfloat16, 128);
    else if (D == 192) GQA_CAST(__nv_bfloat16, 192);
    else return cudaErrorInvalidValue;
  } else {
    if (D == 64) GQA_CAST(__half, 64);
    else if (D == 128) GQA_CAST(__half, 128);
    else if (D == 192) GQA_CAST(__half, 192);
    else return cudaErrorInvalidValue;
  }
#undef GQA_CAST
  return cudaGetLastError();
}

cudaError_t launch_dsink(int B, int Hq, int S, const float* sink, const float* lse, const float* delta,
                         float* dsink, cudaStream_t st) {
  if (Hq <= 0) return cudaSuccess;
  dsink_kernel<<<Hq * kDsinkCluster, kDsinkThreads, 0, st>>>(B, Hq, S, sink, lse, delta, dsink);
  return cudaGetLastError();
}

cudaError_t launch_selftest_wait(int* err, long long limit, cudaStream_t st) {
  selftest_wait_kernel<<<1, 32, 0, st>>>(err, limit);
  return cudaGetLastError();
}

}  // namespace gqa
