// C-ABI entry points of libgqa_attn.so: argument validation, workspace layout,
// TMA tensor-map construction and kernel launches.  See include/gqa_attn.h for
// the contract of each call.
#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>
#include <cuda.h>
#include <cuda_runtime.h>
#include "../../include/gqa_attn.h"
#include "common.cuh"
#include "launch.h"

namespace gqa {
bool kv_kernel_has_dq(int Dqk);
bool kv_kernel_has_bulk_dq(int Dqk);
int kv_kernel_bq(int Dqk);
bool kv_kernel_folds_stats(int Dqk);
}  // namespace gqa

using namespace gqa;

namespace {

constexpr long long kDefaultWaitLimit = 4000000000LL;  // ~2 s of SM clock
std::atomic<long long> g_wait_limit{kDefaultWaitLimit};

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

int num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 148;
  return n;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool supported_dims(int dqk, int dv) {
  return (dqk == 64 && dv == 64) || (dqk == 128 && dv == 128) || (dqk == 192 && dv == 128);
}

bool is_default(const gqa_stride& s) { return s.b == 0 && s.h == 0 && s.s == 0; }

// An explicit layout: 16-byte multiples, rows at least D elements apart, batch stride 0 only for B == 1.
bool valid_stride(const gqa_stride& s, int B, int D) {
  if (is_default(s)) return true;
  if (s.h % 8 || s.s % 8 || s.b % 8) return false;
  if (s.h < D || s.s < D || s.b < 0) return false;
  if (s.b == 0 && B > 1) return false;
  return true;
}

Strides resolve(const gqa_stride& s, int B, int H, int S, int D) {
  if (is_default(s)) return Strides{static_cast<long long>(H) * S * D, static_cast<long long>(S) * D, D};
  // with one batch the batch stride is never used; any valid value keeps the tensor map legal
  return Strides{s.b != 0 ? s.b : static_cast<long long>(H) * S * D, s.h, s.s};
}

gqa_status validate(const gqa_attn_params* p) {
  if (!p) return GQA_ERR_INVALID_ARG;
  if (p->B < 1 || p->Hq < 1 || p->Hkv < 1 || p->S < 0) return GQA_ERR_INVALID_ARG;
  if (p->Hq % p->Hkv != 0) return GQA_ERR_INVALID_ARG;
  if (p->dtype != GQA_F16 && p->dtype != GQA_BF16) return GQA_ERR_INVALID_ARG;
  if (p->causal != 0 && p->causal != 1) return GQA_ERR_INVALID_ARG;
  if (p->window > 0 && !p->causal && p->window_right <= 0) return GQA_ERR_INVALID_ARG;
  if (p->window_right > 0 && p->causal) return GQA_ERR_INVALID_ARG;
  if (!std::isfinite(p->scale) || !(p->scale > 0.f)) return GQA_ERR_INVALID_ARG;
  if (p->Sk < 0 || p->max_seqlen_k < 0) return GQA_ERR_INVALID_ARG;
  if (p->cu_seqlens_k && !p->cu_seqlens) return GQA_ERR_INVALID_ARG;
  if (p->cu_seqlens && !p->cu_seqlens_k && p->Sk != 0 && p->Sk != p->S) return GQA_ERR_INVALID_ARG;
  if (p->S > 0 && (!valid_stride(p->q_st, p->B, p->Dqk) || !valid_stride(p->k_st, p->B, p->Dqk) ||
      !valid_stride(p->v_st, p->B, p->Dv) || !valid_stride(p->o_st, p->B, p->Dv) ||
      !valid_stride(p->do_st, p->B, p->Dv) || !valid_stride(p->dq_st, p->B, p->Dqk) ||
      !valid_stride(p->dk_st, p->B, p->Dqk) || !valid_stride(p->dv_st, p->B, p->Dv)))
    return GQA_ERR_INVALID_ARG;
  if (p->group_mode != GQA_GROUP_TMEM && p->group_mode != GQA_GROUP_ATOMIC) return GQA_ERR_INVALID_ARG;
  if (p->red_mode < GQA_RED_V4 || p->red_mode > GQA_RED_NONE) return GQA_ERR_INVALID_ARG;
  if (p->deterministic != 0 && p->deterministic != 1) return GQA_ERR_INVALID_ARG;
  if (p->cu_seqlens) {
    if (p->B != 1 || p->nseq < 1 || p->nseq > 65535) return GQA_ERR_INVALID_ARG;
    if (p->max_seqlen < 1 || (p->S > 0 && p->max_seqlen > p->S)) return GQA_ERR_INVALID_ARG;
    if (!aligned(p->cu_seqlens, 4)) return GQA_ERR_INVALID_ARG;
  } else if (p->B > 65535) {
    return GQA_ERR_INVALID_ARG;
  }
  if (p->cu_seqlens_k) {
    const int sk = p->Sk > 0 ? p->Sk : p->S;
    if (!aligned(p->cu_seqlens_k, 4) || p->max_seqlen_k < 0 || (sk > 0 && p->max_seqlen_k > sk))
      return GQA_ERR_INVALID_ARG;
  }
  const long long max_len = p->cu_seqlens ? p->max_seqlen : p->S;
  const long long max_len_k = p->cu_seqlens ? (p->cu_seqlens_k && p->max_seqlen_k > 0 ? p->max_seqlen_k : max_len)
                                            : (p->Sk > 0 ? p->Sk : p->S);
  if ((max_len + 127) / 128 > 65535 || (max_len_k + 127) / 128 > 65535) return GQA_ERR_UNSUPPORTED;
  if (!supported_dims(p->Dqk, p->Dv)) return GQA_ERR_UNSUPPORTED;
  // bulk dQ reduction needs shared-memory staging, which only the d=64 tile has room for
  if (!p->deterministic && p->red_mode == GQA_RED_BULK && kv_kernel_has_dq(p->Dqk) && !kv_kernel_has_bulk_dq(p->Dqk))
    return GQA_ERR_UNSUPPORTED;
  return GQA_OK;
}

struct Derived {
  Problem pr;
  WsLayout ws;
  bool need_dq_acc, need_dkdv_acc, group_tmem, need_fold;
};

Derived derive(const gqa_attn_params* p, void* ws) {
  Derived d{};
  d.group_tmem = p->deterministic || p->group_mode == GQA_GROUP_TMEM;
  d.need_dq_acc = !p->deterministic && kv_kernel_has_dq(p->Dqk);
  d.need_dkdv_acc = !d.group_tmem;
  d.need_fold = kv_kernel_folds_stats(p->Dqk);
  Problem& pr = d.pr;
  pr.B = p->B;
  pr.Hq = p->Hq;
  pr.Hkv = p->Hkv;
  pr.S = p->S;
  pr.Dqk = p->Dqk;
  pr.Dv = p->Dv;
  pr.G = p->Hq / p->Hkv;
  pr.causal = p->causal;
  pr.window = p->window > 0 ? p->window : 0;
  pr.right = p->causal ? 1 : (p->window_right > 0 ? p->window_right : 0);
  pr.scale = p->scale;
  pr.scale_log2 = p->scale * kLog2e;
  pr.cu_seqlens = p->cu_seqlens;
  pr.nseqs = p->cu_seqlens ? p->nseq : p->B;
  pr.max_len = p->cu_seqlens ? p->max_seqlen : p->S;
  pr.ntiles = (pr.max_len + kStatTile - 1) / kStatTile;
  pr.wait_limit = g_wait_limit.load();
  pr.Sk = p->Sk > 0 ? p->Sk : p->S;
  pr.cu_seqlens_k = p->cu_seqlens ? p->cu_seqlens_k : nullptr;
  pr.max_len_k = p->cu_seqlens ? (p->cu_seqlens_k && p->max_seqlen_k > 0 ? p->max_seqlen_k : pr.max_len) : pr.Sk;
  pr.q_st = resolve(p->q_st, p->B, p->Hq, p->S, p->Dqk);
  pr.k_st = resolve(p->k_st, p->B, p->Hkv, pr.Sk, p->Dqk);
  pr.v_st = resolve(p->v_st, p->B, p->Hkv, pr.Sk, p->Dv);
  pr.o_st = resolve(p->o_st, p->B, p->Hq, p->S, p->Dv);
  pr.do_st = resolve(p->do_st, p->B, p->Hq, p->S, p->Dv);
  pr.dq_st = resolve(p->dq_st, p->B, p->Hq, p->S, p->Dqk);
  pr.dk_st = resolve(p->dk_st, p->B, p->Hkv, pr.Sk, p->Dqk);
  pr.dv_st = resolve(p->dv_st, p->B, p->Hkv, pr.Sk, p->Dv);
  // packed batches of up to kSchedMaxSeqs sequences: the main kernel takes them longest first
  const bool use_sched = pr.cu_seqlens && pr.nseqs <= kSchedMaxSeqs;
  d.ws = ws_layout(pr.B, pr.Hq, pr.Hkv, pr.S, pr.Sk, pr.Dqk, pr.Dv, pr.nseqs, pr.ntiles, d.need_dq_acc,
                   d.need_dkdv_acc, d.need_fold, use_sched);
  uint8_t* base = static_cast<uint8_t*>(ws);
  pr.err = reinterpret_cast<int*>(base + d.ws.err_off);
  pr.nlse2 = reinterpret_cast<float*>(base + d.ws.lse2_off);
  pr.ndelta = reinterpret_cast<float*>(base + d.ws.delta_off);
  pr.xfold = d.need_fold ? base + d.ws.xf_off : nullptr;
  pr.dq_acc = d.need_dq_acc ? reinterpret_cast<float*>(base + d.ws.dq_off) : nullptr;
  pr.dk_acc = d.need_dkdv_acc ? reinterpret_cast<float*>(base + d.ws.dk_off) : nullptr;
  pr.dv_acc = d.need_dkdv_acc ? reinterpret_cast<float*>(base + d.ws.dv_off) : nullptr;
  pr.sched = (use_sched && base) ? reinterpret_cast<int*>(base + d.ws.sched_off) : nullptr;
  return d;
}

gqa_status check_ws(const gqa_attn_params* p, void* ws, size_t bytes) {
  if (!ws || !aligned(ws, 256)) return GQA_ERR_WORKSPACE;
  if (bytes < gqa_attn_workspace_size(p)) return GQA_ERR_WORKSPACE;
  return GQA_OK;
}

// A 16-bit [B, H, S, D] tensor with element strides st as a 4-D TMA tensor (D, S, H, B); the box is
// 64 columns x box_rows rows of one (b, h), 128-byte swizzled.  Tiles past a head's last row read
// zeros and never cross into another head, whatever the layout.
bool map16(CUtensorMap* m, const void* ptr, int D, int S, int H, int B, const Strides& st, int box_rows, bool bf16) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(S), static_cast<cuuint64_t>(H),
                        static_cast<cuuint64_t>(B)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(st.s) * 2, static_cast<cuuint64_t>(st.h) * 2,
                           static_cast<cuuint64_t>(st.b) * 2};
  cuuint32_t box[4] = {64, static_cast<cuuint32_t>(box_rows), 1, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  return enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4, const_cast<void*>(ptr),
             dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool map32(CUtensorMap* m, const float* ptr, int D, int S, int Z) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(S), static_cast<cuuint64_t>(Z)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 4, static_cast<cuuint64_t>(S) * D * 4};
  cuuint32_t box[3] = {32, 32, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(ptr), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

gqa_status to_status(cudaError_t e) { return e == cudaSuccess ? GQA_OK : GQA_ERR_CUDA; }

}  // namespace

extern "C" {

size_t gqa_attn_params_size(void) { return sizeof(gqa_attn_params); }

size_t gqa_attn_workspace_size(const gqa_attn_params* p) {
  if (validate(p) != GQA_OK) return 0;
  return derive(p, nullptr).ws.total;
}

gqa_status gqa_attn_fwd(const gqa_attn_params* p, const void* q, const void* k, const void* v, const float* sink,
                        void* o, float* lse, void* workspace, size_t ws_bytes, void* stream) {
  gqa_status s = validate(p);
  if (s != GQA_OK) return s;
  if ((s = check_ws(p, workspace, ws_bytes)) != GQA_OK) return s;
  if (!q || !k || !v || !o || !lse) return GQA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(lse, 4) ||
      (sink && !aligned(sink, 4)))
    return GQA_ERR_INVALID_ARG;
  if (p->S == 0) return GQA_OK;
  Derived d = derive(p, workspace);
  const bool bf = p->dtype == GQA_BF16;
  Maps m;
  std::memset(&m, 0, sizeof(m));
  const int bk = fwd_kernel_bk(p->Dqk);
  if (!map16(&m.q, q, p->Dqk, p->S, p->Hq, p->B, d.pr.q_st, 128, bf) || !map16(&m.k, k, p->Dqk, d.pr.Sk, p->Hkv, p->B, d.pr.k_st, bk, bf) ||
      !map16(&m.v, v, p->Dv, d.pr.Sk, p->Hkv, p->B, d.pr.v_st, bk, bf))
    return GQA_ERR_CUDA;
  return to_status(launch_fwd(d.pr, bf, m, sink, o, lse, static_cast<cudaStream_t>(stream)));
}

gqa_status gqa_attn_bwd_preprocess(const gqa_attn_params* p, const void* o, const void* dout, const float* lse,
                                   float* delta, void* workspace, size_t ws_bytes, void* stream) {
  gqa_status s = validate(p);
  if (s != GQA_OK) return s;
  if ((s = check_ws(p, workspace, ws_bytes)) != GQA_OK) return s;
  if (!o || !dout || !lse || !delta) return GQA_ERR_INVALID_ARG;
  if (!aligned(o, 16) || !aligned(dout, 16) || !aligned(lse, 4) || !aligned(delta, 4)) return GQA_ERR_INVALID_ARG;
  if (p->S == 0) return GQA_OK;
  Derived d = derive(p, workspace);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (d.need_dkdv_acc) {  // the dK / dV accumulators span the key axis: zeroed here, not per query row
    const size_t rows = static_cast<size_t>(p->B) * p->Hkv * d.pr.Sk;
    if (cudaMemsetAsync(d.pr.dk_acc, 0, rows * p->Dqk * 4, st) != cudaSuccess ||
        cudaMemsetAsync(d.pr.dv_acc, 0, rows * p->Dv * 4, st) != cudaSuccess)
      return GQA_ERR_CUDA;
  }
  return to_status(launch_preprocess(d.pr, p->dtype == GQA_BF16, o, dout, lse, delta, d.need_dq_acc,
                                     num_sms(), st));
}

gqa_status gqa_attn_bwd(const gqa_attn_params* p, const void* q, const void* k, const void* v, const void* dout,
                        void* dq, void* dk, void* dv, void* workspace, size_t ws_bytes, void* stream) {
  gqa_status s = validate(p);
  if (s != GQA_OK) return s;
  if ((s = check_ws(p, workspace, ws_bytes)) != GQA_OK) return s;
  Derived d = derive(p, workspace);
  const bool dq_pass = !d.need_dq_acc;  // deterministic, or dims whose dQ always comes from that pass
  if (!q || !k || !v || !dout) return GQA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(dout, 16)) return GQA_ERR_INVALID_ARG;
  if (dq_pass && (!dq || !aligned(dq, 16))) return GQA_ERR_INVALID_ARG;
  if (d.group_tmem && (!dk || !dv || !aligned(dk, 16) || !aligned(dv, 16))) return GQA_ERR_INVALID_ARG;
  if (p->S == 0) return GQA_OK;
  const bool bf = p->dtype == GQA_BF16;
  const int bq = kv_kernel_bq(p->Dqk);
  Maps m;
  std::memset(&m, 0, sizeof(m));
  if (!map16(&m.q, q, p->Dqk, p->S, p->Hq, p->B, d.pr.q_st, bq, bf) || !map16(&m.dout, dout, p->Dv, p->S, p->Hq, p->B, d.pr.do_st, bq, bf) ||
      !map16(&m.k, k, p->Dqk, d.pr.Sk, p->Hkv, p->B, d.pr.k_st, 128, bf) || !map16(&m.v, v, p->Dv, d.pr.Sk, p->Hkv, p->B, d.pr.v_st, 128, bf))
    return GQA_ERR_CUDA;
  if (d.need_dq_acc && !map32(&m.dq_acc, d.pr.dq_acc, p->Dqk, p->S, p->B * p->Hq)) return GQA_ERR_CUDA;
  if (d.need_dkdv_acc && (!map32(&m.dk_acc, d.pr.dk_acc, p->Dqk, d.pr.Sk, p->B * p->Hkv) ||
                          !map32(&m.dv_acc, d.pr.dv_acc, p->Dv, d.pr.Sk, p->B * p->Hkv)))
    return GQA_ERR_CUDA;
  static const int red_to_mode[4] = {kDqRedV4, kDqBulk, kDqScalar, kDqStore};
  KvLaunch kl;
  kl.group_tmem = d.group_tmem ? 1 : 0;
  kl.dq_mode = d.need_dq_acc ? red_to_mode[p->red_mode] : kDqNone;
  kl.kv_red_mode = red_to_mode[p->red_mode];
  kl.dk = dk;
  kl.dv = dv;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = launch_bwd_kv(d.pr, bf, m, kl, st);
  if (e != cudaSuccess) return GQA_ERR_CUDA;
  if (dq_pass) {
    Maps m2 = m;  // the query-stationary pass: 128-row Q / dO boxes, K / V boxes of its key tile
    const int bk = q_kernel_bk();
    if (!map16(&m2.q, q, p->Dqk, p->S, p->Hq, p->B, d.pr.q_st, 128, bf) ||
        !map16(&m2.dout, dout, p->Dv, p->S, p->Hq, p->B, d.pr.do_st, 128, bf) ||
        !map16(&m2.k, k, p->Dqk, d.pr.Sk, p->Hkv, p->B, d.pr.k_st, bk, bf) || !map16(&m2.v, v, p->Dv, d.pr.Sk, p->Hkv, p->B, d.pr.v_st, bk, bf))
      return GQA_ERR_CUDA;
    e = launch_dq(d.pr, bf, m2, dq, st);
    if (e != cudaSuccess) return GQA_ERR_CUDA;
  }
  return GQA_OK;
}

gqa_status gqa_attn_bwd_postprocess(const gqa_attn_params* p, void* dq, void* dk, void* dv, void* workspace,
                                    size_t ws_bytes, void* stream) {
  gqa_status s = validate(p);
  if (s != GQA_OK) return s;
  if ((s = check_ws(p, workspace, ws_bytes)) != GQA_OK) return s;
  Derived d = derive(p, workspace);
  if (d.need_dq_acc && (!dq || !aligned(dq, 16))) return GQA_ERR_INVALID_ARG;
  if (d.need_dkdv_acc && (!dk || !dv || !aligned(dk, 16) || !aligned(dv, 16))) return GQA_ERR_INVALID_ARG;
  if (p->S == 0) return GQA_OK;
  const bool bf = p->dtype == GQA_BF16;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int sms = num_sms();
  if (d.need_dq_acc) {
    cudaError_t e = launch_cast(d.pr.dq_acc, dq, p->B, p->Hq, p->S, p->Dqk, d.pr.dq_st, p->scale, bf, sms, st);
    if (e != cudaSuccess) return GQA_ERR_CUDA;
  }
  if (d.need_dkdv_acc) {
    cudaError_t e = launch_cast(d.pr.dk_acc, dk, p->B, p->Hkv, d.pr.Sk, p->Dqk, d.pr.dk_st, p->scale, bf, sms, st);
    if (e == cudaSuccess) e = launch_cast(d.pr.dv_acc, dv, p->B, p->Hkv, d.pr.Sk, p->Dv, d.pr.dv_st, 1.f, bf, sms, st);
    if (e != cudaSuccess) return GQA_ERR_CUDA;
  }
  return GQA_OK;
}

gqa_status gqa_attn_dsink(const gqa_attn_params* p, const float* sink, const float* lse, const float* delta,
                          float* dsink, void* stream) {
  gqa_status s = validate(p);
  if (s != GQA_OK) return s;
  if (!sink || !lse || !delta || !dsink) return GQA_ERR_INVALID_ARG;
  if (!aligned(sink, 4) || !aligned(lse, 4) || !aligned(delta, 4) || !aligned(dsink, 4)) return GQA_ERR_INVALID_ARG;
  return to_status(launch_dsink(p->B, p->Hq, p->S, sink, lse, delta, dsink, static_cast<cudaStream_t>(stream)));
}

gqa_status gqa_attn_get_device_error(void* workspace, size_t ws_bytes, void* stream, int* site) {
  if (site) *site = 0;
  if (!workspace || ws_bytes < 256 || !aligned(workspace, 256)) return GQA_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return GQA_ERR_CUDA;
  int word = 0;
  if (cudaMemcpy(&word, workspace, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return GQA_ERR_CUDA;
  if (word != 0) {
    const int zero = 0;
    if (cudaMemcpy(workspace, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return GQA_ERR_CUDA;
  }
  if (site) *site = word;
  if (word == 0) return GQA_OK;
  if (static_cast<unsigned>(word) & 0x80000000u) return GQA_ERR_DEVICE_TIMEOUT;
  return GQA_ERR_DEVICE_INPUT;
}

void gqa_attn_set_wait_limit(long long cycles) {
  g_wait_limit.store(cycles > 0 ? cycles : kDefaultWaitLimit);
}

gqa_status gqa_attn_selftest_wait_timeout(void* workspace, size_t ws_bytes, void* stream) {
  if (!workspace || ws_bytes < 256 || !aligned(workspace, 256)) return GQA_ERR_WORKSPACE;
  return to_status(
      launch_selftest_wait(static_cast<int*>(workspace), g_wait_limit.load(), static_cast<cudaStream_t>(stream)));
}

const char* gqa_attn_strerror(gqa_status s) {
  switch (s) {
    case GQA_OK: return "ok";
    case GQA_ERR_INVALID_ARG: return "invalid argument";
    case GQA_ERR_UNSUPPORTED: return "unsupported problem";
    case GQA_ERR_WORKSPACE: return "workspace missing, too small or misaligned";
    case GQA_ERR_CUDA: return "CUDA error";
    case GQA_ERR_DEVICE_TIMEOUT: return "a device-side wait timed out";
    case GQA_ERR_DEVICE_INPUT: return "device-side input check failed";
  }
  return "unknown status";
}

}  // extern "C"

// ---------------------------------------------------------------- no-allocation backward
// Some callers cannot call cudaMalloc: code that runs while a CUDA graph is being
// captured with a relaxed/global capture mode that forbids allocation, allocators
// that own the whole device pool, and embedded runtimes whose memory is fixed at
// start-up.  For them gqa_attn_bwd_noalloc runs the backward with its scratch in
// the file-scope device array below instead of a caller workspace.  The array is
// part of the library's device image: every GPU that loads the library holds
// these bytes until the process exits.
namespace {
constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;  // 16 MiB
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];
constexpr int kNoAllocMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kNoAllocMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once per
// device; the host-side symbol is only a stand-in and must never reach a kernel).
gqa_status noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNoAllocMaxDevices) return GQA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return GQA_ERR_CUDA;
    g_noalloc_ptr[dev] = ptr;
  }
  *out = g_noalloc_ptr[dev];
  return GQA_OK;
}
}  // namespace

extern "C" gqa_status gqa_attn_bwd_noalloc(const gqa_attn_params* p, const void* q, const void* k, const void* v,
                                           const void* o, const void* dout, const float* lse, float* delta, void* dq,
                                           void* dk, void* dv, void* stream) {
  gqa_status s = validate(p);
  if (s != GQA_OK) return s;
  if (gqa_attn_workspace_size(p) > kNoAllocScratchBytes) return GQA_ERR_WORKSPACE;
  void* scratch = nullptr;
  if ((s = noalloc_scratch(&scratch)) != GQA_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // the error word must start at zero; the other regions are fully rewritten by the preprocess
  if (cudaMemsetAsync(scratch, 0, 256, st) != cudaSuccess) return GQA_ERR_CUDA;
  if ((s = gqa_attn_bwd_preprocess(p, o, dout, lse, delta, scratch, kNoAllocScratchBytes, stream)) != GQA_OK) return s;
  if ((s = gqa_attn_bwd(p, q, k, v, dout, dq, dk, dv, scratch, kNoAllocScratchBytes, stream)) != GQA_OK) return s;
  return gqa_attn_bwd_postprocess(p, dq, dk, dv, scratch, kNoAllocScratchBytes, stream);
}

// The error word of the scratch array: device-side failures of gqa_attn_bwd_noalloc (a packed
// sequence longer than max_seqlen, malformed cu_seqlens, a wait that timed out) are recorded there,
// and a caller without a workspace of its own reads them back through this call.
extern "C" gqa_status gqa_attn_noalloc_get_device_error(void* stream, int* site) {
  if (site) *site = 0;
  void* scratch = nullptr;
  gqa_status s = noalloc_scratch(&scratch);
  if (s != GQA_OK) return s;
  return gqa_attn_get_device_error(scratch, kNoAllocScratchBytes, stream, site);
}
