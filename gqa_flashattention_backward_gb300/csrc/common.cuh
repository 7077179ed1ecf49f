// Shared definitions of the CUDA path: the problem descriptor handed to every
// kernel, the workspace layout, and sequence/tile bookkeeping.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace gqa {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kStatTile = 128;  // row statistics are stored in blocks of 128 query rows

// Error-word codes (low bits); bit 31 marks a timed-out wait.
enum : int {
  kErrSeqTooLong = 0x40000001,
  kErrBadSeqlens = 0x40000002,
};

// Element strides of a 16-bit [B, H, S, D] tensor (head-dim stride 1), resolved on the host.
struct Strides {
  long long b, h, s;
  __host__ __device__ __forceinline__ long long row(int bi, int hi, long long si) const {
    return bi * b + hi * h + si * s;
  }
};

// Everything a kernel needs to know about the attention problem.
struct Problem {
  int B, Hq, Hkv, S, Dqk, Dv, G;  // G = Hq / Hkv
  int causal, window;
  int right;          // right extent: keys with j - (i + off) < right; 1 = causal, <= 0 = unlimited
  float scale;        // softmax scale
  float scale_log2;   // scale * log2(e): logits are exponentiated with ex2
  const int32_t* cu_seqlens;  // device [nseqs+1] or null (dense)
  int nseqs;          // packed sequences, or B when dense
  int max_len;        // longest sequence (S when dense)
  int ntiles;         // ceil(max_len / 128): stat tiles per (head, sequence)
  int* err;           // device error word (workspace)
  long long wait_limit;
  // workspace regions
  float* nlse2;       // [Hq][nseqs][ntiles][128]  -LSE * log2(e), -inf on padding rows
  float* ndelta;      // same layout, -Delta, 0 on padding rows (both negated so the
                      // kernels use one packed fma / add per pair of elements)
  uint8_t* xfold;     // or null: [Hq][nseqs][ntiles] 4 KB tiles, one 32-byte bf16 row per query:
                      // -LSE/scale and -Delta, each split hi + mid + lo, in the tensor core's
                      // no-swizzle K-major layout (the main kernel adds them with an MMA)
  float* dq_acc;      // [B][Hq][S][Dqk] fp32
  float* dk_acc;      // [B][Hkv][S][Dqk] fp32
  float* dv_acc;      // [B][Hkv][S][Dv] fp32
  // layouts of the caller's 16-bit tensors (element offset of row (b, h, s) = row(b, h, s))
  Strides q_st, k_st, v_st, o_st, do_st, dq_st, dk_st, dv_st;
  // keys: rows per batch (or packed key tokens), device key offsets (or null: cu_seqlens), longest
  int Sk;
  const int32_t* cu_seqlens_k;
  int max_len_k;
  // packed batches: the main kernel's sequence order, longest first, written by the preprocess (null:
  // the packing order)
  int* sched;
};

// One sequence of the (possibly packed) batch.
struct Seq {
  int b;      // batch index (0 when packed)
  int start;  // first token on the S axis
  int len;    // tokens
};

__device__ __forceinline__ bool load_seq(const Problem& p, int s, Seq& q) {
  if (p.cu_seqlens) {
    const int a = __ldg(p.cu_seqlens + s), e = __ldg(p.cu_seqlens + s + 1);
    q.b = 0;
    q.start = a;
    q.len = e - a;
    if (q.len < 0 || a < 0 || e > p.S) {
      atomicCAS(p.err, 0, kErrBadSeqlens);
      q.len = 0;
      return false;
    }
    if (q.len > p.max_len) {
      atomicCAS(p.err, 0, kErrSeqTooLong);
      q.len = 0;
      return false;
    }
  } else {
    q.b = s;
    q.start = 0;
    q.len = p.S;
  }
  return true;
}

// The keys of sequence s (same checks as load_seq, against the key axis).
__device__ __forceinline__ bool load_kseq(const Problem& p, int s, Seq& k) {
  const int32_t* cu = p.cu_seqlens_k ? p.cu_seqlens_k : p.cu_seqlens;
  if (cu) {
    const int a = __ldg(cu + s), e = __ldg(cu + s + 1);
    k.b = 0;
    k.start = a;
    k.len = e - a;
    if (k.len < 0 || a < 0 || e > p.Sk) {
      atomicCAS(p.err, 0, kErrBadSeqlens);
      k.len = 0;
      return false;
    }
    if (k.len > p.max_len_k) {
      atomicCAS(p.err, 0, kErrSeqTooLong);
      k.len = 0;
      return false;
    }
  } else {
    k.b = s;
    k.start = 0;
    k.len = p.Sk;
  }
  return true;
}

// Visibility of key j (local) to query i (local) is decided on the pair's diagonal distance
// d = i + off - j, off = Lk - Lq aligning the causal diagonal at the bottom right (0 when a sequence
// has as many keys as queries): the key exists, d > -right (right = 1: causal) and d < window.
// The tile loops hoist everything but a compile-time offset into d: two comparisons per element.
__device__ __forceinline__ bool visible_d(int d, bool key_exists, int right, int window) {
  return key_exists && (right <= 0 || d > -right) && (window <= 0 || d < window);
}

// ---------------------------------------------------------------- longest-first sequence order
// The main kernel's grid runs sequence by sequence (each sequence's KV tiles together, so its query
// tiles stay in L2 while they are read), tile 0 -- the heaviest under a causal mask -- first.  For
// packed batches the preprocess writes the order of the sequences, longest (most KV tiles) first, so
// short sequences fill the last wave instead of a long one arriving last: perm[slot] = sequence.
constexpr int kSchedMaxSeqs = 256;  // sequences the one-block sort orders

// perm[rank] = q for the sequences q < n ranked by key[q] (KV tiles), largest first, ties by index;
// run by threads tid < nth of one block (or one host thread, nth = 1).
__host__ __device__ inline void sched_fill(int* perm, const int* key, int n, int tid, int nth) {
  for (int q = tid; q < n; q += nth) {
    int rank = 0;
    for (int t = 0; t < n; ++t) rank += (key[t] > key[q]) || (key[t] == key[q] && t < q);
    perm[rank] = q;
  }
}

// Index of the first float of a stats tile: head h, sequence s, 128-row tile t.
__host__ __device__ __forceinline__ size_t stat_index(const Problem& p, int h, int s, int t) {
  return ((static_cast<size_t>(h) * p.nseqs + s) * p.ntiles + t) * kStatTile;
}

// ---------------------------------------------------------------- workspace
struct WsLayout {
  size_t err_off, lse2_off, delta_off, xf_off, dq_off, dk_off, dv_off, sched_off, total;
};

constexpr int kFoldRowBytes = 32;  // 16 bf16 values per query row in an xfold tile

__host__ inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

__host__ inline WsLayout ws_layout(int B, int Hq, int Hkv, int S, int Sk, int Dqk, int Dv, int nseqs, int ntiles,
                                   bool need_dq_acc, bool need_dkdv_acc, bool need_fold, bool need_sched = false) {
  WsLayout w{};
  size_t off = 0;
  w.err_off = off;
  off += 256;
  const size_t nstat = static_cast<size_t>(Hq) * nseqs * ntiles * kStatTile;
  w.lse2_off = off;
  off = align256(off + nstat * 4);
  w.delta_off = off;
  off = align256(off + nstat * 4);
  w.xf_off = off;
  if (need_fold) off = align256(off + nstat * kFoldRowBytes);
  w.dq_off = off;
  if (need_dq_acc) off = align256(off + static_cast<size_t>(B) * Hq * S * Dqk * 4);
  w.dk_off = off;
  if (need_dkdv_acc) off = align256(off + static_cast<size_t>(B) * Hkv * Sk * Dqk * 4);
  w.dv_off = off;
  if (need_dkdv_acc) off = align256(off + static_cast<size_t>(B) * Hkv * Sk * Dv * 4);
  w.sched_off = off;
  if (need_sched) off = align256(off + static_cast<size_t>(nseqs) * 4);
  w.total = off;
  return w;
}

// ---------------------------------------------------------------- tile ranges
// (len_q queries and len_k keys in the sequence; off = len_k - len_q; see `visible`)

// Query rows that can see some key of the 128-row KV tile kt, as a range of query tiles of
// `bq` rows: [*t0, *t1).
__host__ __device__ __forceinline__ void q_tiles_for_kv_tile(int kt, int len_q, int len_k, int bq, int right,
                                                             int window, int* t0, int* t1) {
  const int ntq = (len_q + bq - 1) / bq;
  const long long off = static_cast<long long>(len_k) - len_q;
  const long long j_lo = static_cast<long long>(kt) * 128;
  const long long i_first = right > 0 ? j_lo - off - right + 1 : 0;  // first row reaching the tile
  int a = i_first > 0 ? static_cast<int>(i_first / bq) : 0;
  if (a > ntq) a = ntq;
  int b = ntq;
  if (window > 0) {
    const long long i_hi = j_lo + 127 + window - 1 - off;  // last row seeing key j_lo + 127
    const long long tb = i_hi < 0 ? 0 : i_hi / bq + 1;
    if (tb < b) b = static_cast<int>(tb);
  }
  *t0 = a;
  *t1 = b > a ? b : a;
}

// Key tiles of `bk` rows visible to the query tile qt of 128 rows: [*k0, *k1).
__host__ __device__ __forceinline__ void kv_tiles_for_q_tile(int qt, int len_q, int len_k, int bk, int right,
                                                             int window, int* k0, int* k1) {
  const int ntk = (len_k + bk - 1) / bk;
  const long long off = static_cast<long long>(len_k) - len_q;
  const long long d_lo = static_cast<long long>(qt) * 128 + off, d_hi = d_lo + 127;  // diagonals of the tile
  int b = ntk;
  if (right > 0) {
    const long long j_hi = d_hi + right - 1;  // last key the tile's last row sees
    b = j_hi < 0 ? 0 : (j_hi / bk + 1 < ntk ? static_cast<int>(j_hi / bk + 1) : ntk);
  }
  int a = 0;
  if (window > 0) {
    const long long j_lo = d_lo - window + 1;
    a = j_lo > 0 ? static_cast<int>(j_lo / bk) : 0;
  }
  *k0 = a;
  *k1 = b > a ? b : a;
}

}  // namespace gqa
