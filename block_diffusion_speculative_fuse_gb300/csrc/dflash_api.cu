// C ABI: argument checks, TMA descriptors, workspace layout and the launch
// sequences of the draft step, the context fuse / K-V injection, greedy
// verify and the causal target forward.  Host code only; every arithmetic
// step runs in the kernels of this library.
#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>
#include <vector>

#include "dflash.h"
#include "kernels.h"

using namespace dflash;

namespace {

thread_local int g_last_cuda = 0;

int cuda_fail(cudaError_t e) {
  g_last_cuda = static_cast<int>(e);
  return DFLASH_ERR_CUDA;
}
#define DF_CUDA(expr)                               \
  do {                                              \
    cudaError_t e__ = (expr);                       \
    if (e__ != cudaSuccess) return cuda_fail(e__);  \
  } while (0)

// ---------------------------------------------------------------- driver entry
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

int load_encode() {
  if (g_encode != nullptr) return DFLASH_OK;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                   cudaEnableDefault, &q);
  if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || fn == nullptr)
    return DFLASH_ERR_NO_DEVICE;
  g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  return DFLASH_OK;
}

// 2-D bf16 map over [rows][cols] (row stride ld elements), box [box_rows][64],
// 128-byte swizzle, zero fill out of bounds.
int encode_map(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint64_t ld,
               uint32_t box_rows) {
  if ((reinterpret_cast<uintptr_t>(base) & 15) != 0 || (ld * 2) % 16 != 0)
    return DFLASH_ERR_INVALID_ARG;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {ld * 2};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(kTileK), box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? DFLASH_OK : DFLASH_ERR_INVALID_ARG;
}

// 3-D bf16 map over [rows][d] (d = 64 or 128): dims (64 columns, row, d/64
// column halves), box (64, 16, d/64): 16 rows of both column halves as
// [half][16 rows][128 B], 128-byte swizzled, zero fill out of bounds.
int encode_map_rows16(CUtensorMap* map, const void* base, uint64_t rows, uint32_t d) {
  if ((reinterpret_cast<uintptr_t>(base) & 15) != 0 || (d != 64 && d != 128))
    return DFLASH_ERR_INVALID_ARG;
  cuuint64_t dims[3] = {64, rows, d / 64};
  cuuint64_t strides[2] = {d * 2ull, 128ull};
  cuuint32_t box[3] = {64, 16, d / 64};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? DFLASH_OK : DFLASH_ERR_INVALID_ARG;
}

// 2-D uint8 map over [rows][cols] bytes (cols a multiple of 16), box
// [box_rows][cols], no swizzle, zero fill out of bounds.
int encode_map_u8(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                  uint32_t box_rows) {
  if ((reinterpret_cast<uintptr_t>(base) & 15) != 0 || cols % 16 != 0 || cols > 256)
    return DFLASH_ERR_INVALID_ARG;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(cols), box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? DFLASH_OK : DFLASH_ERR_INVALID_ARG;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace

struct dflash_model_s {
  dflash_config cfg;
  dflash_weights w;
  int device = 0;
  int sms = 148;
  bool is_draft = false;
  bool attn_tc = true;      // drafter attention on tcgen05 (attention_tc05.cu) when the shape allows
  int two_term_layers = -1;  // layers [0, k) carry two-term (hi + lo) activations; -1: automatic
  // GEMM: k-blocks its producer still has to request when the next kernel
  // may launch (< 0: at the start)
  int dep_lead = 2;
  int pre_mask = 15;  // GEMM epilogue inputs loaded during the main loop (GemmParams::pre_mask)
  CUtensorMap m_wqkv, m_wo, m_gu, m_down, m_lm, m_fc;
  float2 rope[kMaxRopePairs];
  int qkv_rows = 0, q_dim = 0, kv_dim = 0;
};

namespace {

// Workspace header (zeroed by dflash_workspace_init; every kernel leaves
// what it uses at zero): [0, 256) status word (int32 [0] code, [1] site, [2]
// LM-head argmax ticket), [256, 32 KiB) split-K counters, [32 KiB, 64 KiB)
// LM-head argmax keys (uint64 per row).
constexpr size_t kHeaderBytes = 64 * 1024;
constexpr size_t kAmaxKeyOff = 32 * 1024;
constexpr int kMaxCounters = (kAmaxKeyOff - 256) / 4;
constexpr int kMaxAmaxKeyRows = static_cast<int>((kHeaderBytes - kAmaxKeyOff) / 8);
constexpr int kTargetSplitKeys = 512;
constexpr int kMaxClusterSplits = 8;  // portable cluster size

size_t al256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

const uint16_t* u16(const void* p) { return static_cast<const uint16_t*>(p); }

// Split-K count: enough CTAs for one resident wave, at least 2 k-blocks per
// split.  For a target (batch-invariant path) it depends on the weight shape
// only, never on the number of activation rows.
int choose_splits(const dflash_model_s* m, int n_tiles, int m_tiles, int kb_total, int bn) {
  // resident CTAs per SM of the GEMM (shared-memory bound): 3 for BN <= 32
  const int per_sm = bn <= 32 ? 3 : bn <= 128 ? 2 : 1;
  const int capacity = m->sms * (m->is_draft ? per_sm : 2);
  const int base = n_tiles * (m->is_draft ? m_tiles : 1);
  int s = capacity / std::max(1, base);
  s = std::max(1, std::min(s, kb_total / 2));
  s = std::min(s, kMaxClusterSplits);  // the splits of a tile form one thread-block cluster
  return s;
}

struct Ws {
  uint8_t* base = nullptr;
  size_t off = kHeaderBytes;
  size_t cap = 0;
  bool dry = false;
  template <typename T>
  T* take(size_t n) {
    T* p = dry ? nullptr : reinterpret_cast<T*>(base + off);
    off = al256(off + n * sizeof(T));
    return p;
  }
  int32_t* status() const { return dry ? nullptr : reinterpret_cast<int32_t*>(base); }
  int32_t* counters() const { return dry ? nullptr : reinterpret_cast<int32_t*>(base + 256); }
  unsigned long long* amax_keys() const {
    return dry ? nullptr : reinterpret_cast<unsigned long long*>(base + kAmaxKeyOff);
  }
};

// Buffers of one stack pass over `rows` activation rows (+ ctx rows on the QKV input).
struct StackBufs {
  float* x;
  uint16_t* a;     // [rows + ctx][H]
  uint16_t* q;     // [rows][hq][d]
  uint16_t* kblk;
  uint16_t* vblk;
  float* o_part;
  float* ml_part;
  uint16_t* o;     // [rows][q_dim]
  uint16_t* a2;    // [rows][H]
  uint16_t* hmid;  // [rows][F]
  // low bf16 halves of o, a2, hmid: the O-projection, gate/up and down GEMMs
  // multiply the two-term expansion hi + lo of their activation operand
  uint16_t* o_lo;
  uint16_t* a2_lo;
  uint16_t* hmid_lo;
  float* partial;
  float* amax_val;
  int32_t* amax_idx;
  float* ctx_f32;
  float* ssq_a;    // [rows][H/128] per-tile sums of squares of the rows behind `a`
  float* ssq_a2;   // same for `a2`
};

struct GemmShape {
  int N, K, m_rows;
};

size_t partial_floats(const dflash_model_s* m, int rows_main, int rows_qkv) {
  const dflash_config& c = m->cfg;
  const GemmShape shapes[6] = {{m->qkv_rows, c.hidden, rows_qkv},
                               {2 * m->kv_dim, c.hidden, rows_qkv},
                               {c.hidden, m->q_dim, rows_main},
                               {2 * c.mlp, c.hidden, rows_main},
                               {c.hidden, c.mlp, rows_main},
                               {c.hidden, c.n_taps * c.hidden, rows_qkv}};
  size_t mx = 0;
  for (const GemmShape& g : shapes) {
    if (g.K <= 0 || g.N <= 0 || g.m_rows <= 0) continue;
    const int bn = gemm_bn_for(g.m_rows, g.N, m->sms);
    const int mt = (g.m_rows + bn - 1) / bn;
    const int s = choose_splits(m, g.N / kTileN, mt, g.K / kTileK, bn);
    // splits up to the cluster size reduce through DSMEM and need no buffer
    if (s > kMaxClusterSplits) mx = std::max(mx, static_cast<size_t>(s) * g.m_rows * g.N);
  }
  return mx;
}

// Keys per attention split.  Drafter: at most kMaxAttnCluster-1 context
// splits + the block split, so the splits of a query tile fit one cluster and
// combine through DSMEM.  Target: a fixed 512 (split boundaries independent
// of the batch).
int attn_split_keys(const dflash_model_s* m, int batch, int max_keys) {
  (void)batch;
  if (!m->is_draft) return kTargetSplitKeys;
  const int nc = kMaxAttnCluster - 1;
  long long s = (static_cast<long long>(max_keys) + nc - 1) / nc;
  s = ((s + 63) / 64) * 64;
  // a split's page list must fit the staged page ids (kMaxSplitPages)
  s = std::min<long long>(s, 8128);
  return static_cast<int>(std::max<long long>(64, s));
}
int attn_n_splits(const dflash_model_s* m, int split_keys, int max_keys) {
  const int n = (max_keys + split_keys - 1) / split_keys;
  return m->is_draft ? n + 1 : std::max(1, n);
}


void layout_stack(const dflash_model_s* m, Ws& ws, StackBufs& b, int batch, int n, int ctx_rows,
                  int max_keys) {
  const dflash_config& c = m->cfg;
  const int rows = batch * n;
  b.x = ws.take<float>(static_cast<size_t>(rows) * c.hidden);
  b.a = ws.take<uint16_t>(static_cast<size_t>(rows + ctx_rows) * c.hidden);
  b.q = ws.take<uint16_t>(static_cast<size_t>(rows) * m->q_dim);
  b.kblk = ws.take<uint16_t>(static_cast<size_t>(rows) * m->kv_dim);
  b.vblk = ws.take<uint16_t>(static_cast<size_t>(rows) * m->kv_dim);
  const int sk = attn_split_keys(m, batch, max_keys);
  const int ns = attn_n_splits(m, sk, max_keys);
  b.o_part = ws.take<float>(static_cast<size_t>(ns) * rows * c.n_q_heads * c.head_dim);
  b.ml_part = ws.take<float>(static_cast<size_t>(ns) * rows * c.n_q_heads * 2);
  b.o = ws.take<uint16_t>(static_cast<size_t>(rows) * m->q_dim);
  b.a2 = ws.take<uint16_t>(static_cast<size_t>(rows) * c.hidden);
  b.hmid = ws.take<uint16_t>(static_cast<size_t>(rows) * c.mlp);
  b.o_lo = ws.take<uint16_t>(static_cast<size_t>(rows) * m->q_dim);
  b.a2_lo = ws.take<uint16_t>(static_cast<size_t>(rows) * c.hidden);
  b.hmid_lo = ws.take<uint16_t>(static_cast<size_t>(rows) * c.mlp);
  b.partial = ws.take<float>(partial_floats(m, rows, rows + ctx_rows));
  const int vt = c.vocab / kTileN;
  b.amax_val = ws.take<float>(static_cast<size_t>(rows) * vt);
  b.amax_idx = ws.take<int32_t>(static_cast<size_t>(rows) * vt);
  b.ctx_f32 = nullptr;
  b.ssq_a = ws.take<float>(static_cast<size_t>(rows) * (c.hidden / kTileN));
  b.ssq_a2 = ws.take<float>(static_cast<size_t>(rows) * (c.hidden / kTileN));
}

GemmParams gemm_base(const dflash_model_s* m, int M, int N, int K, int bn, Ws& ws) {
  GemmParams p;
  std::memset(&p, 0, sizeof(p));
  p.M = M;
  p.N = N;
  p.K = K;
  p.w_tile_step = kTileN;
  p.w_half_gap = 64;
  p.kb_total = K / kTileK;
  const int mt = (M + bn - 1) / bn;
  p.splits = choose_splits(m, N / kTileN, mt, p.kb_total, bn);
  p.kb_per_split = (p.kb_total + p.splits - 1) / p.splits;
  p.splits = (p.kb_total + p.kb_per_split - 1) / p.kb_per_split;
  p.counters = ws.counters();
  p.status = ws.status();
  p.dep_lead = m->dep_lead;
  p.pre_mask = m->pre_mask;
  return p;
}


// x_lo (optional): low bf16 halves of the activation operand, same layout as x.
int run_gemm(const dflash_model_s* m, const CUtensorMap* wmap, const void* x, int ld_x,
             GemmParams& p, float* partial, cudaStream_t s, const void* x_lo = nullptr) {
  const int bn = gemm_bn_for(p.M, p.N, m->sms);
  const int mt = (p.M + bn - 1) / bn;
  p.cluster = 0;
  if (p.splits > 1) {
    // split-K partials are reduced through distributed shared memory inside a
    // cluster of the tile's splits (measured faster than a global-memory
    // reduction even when the clusters run in more than one wave)
    p.cluster = p.splits <= kMaxClusterSplits ? 1 : 0;
    if (!p.cluster) {
      if ((p.N / kTileN) * mt > kMaxCounters) return DFLASH_ERR_CAPACITY;
      p.partial = partial;
    }
  }
  CUtensorMap xmap, xmap_lo;
  int rc = encode_map(&xmap, x, p.M, p.K, ld_x, bn);
  if (!rc && x_lo != nullptr) rc = encode_map(&xmap_lo, x_lo, p.M, p.K, ld_x, bn);
  if (rc) return rc;
  DF_CUDA(gemm_launch(wmap, &xmap, x_lo != nullptr ? &xmap_lo : nullptr, p, bn, s, true));
  return DFLASH_OK;
}

QkvEpi qkv_base(const dflash_model_s* m, int layer) {
  const dflash_config& c = m->cfg;
  QkvEpi e;
  std::memset(&e, 0, sizeof(e));
  e.n_q_heads = c.n_q_heads;
  e.n_kv_heads = c.n_kv_heads;
  e.head_dim = c.head_dim;
  e.eps = c.rms_eps;
  if (c.qk_norm) {
    e.q_norm = u16(m->w.q_norm) + static_cast<size_t>(layer) * c.head_dim;
    e.k_norm = u16(m->w.k_norm) + static_cast<size_t>(layer) * c.head_dim;
  }
  e.page_size = c.page_size;
  std::memcpy(e.rope, m->rope, sizeof(e.rope));
  return e;
}

int kv_terms_of(const dflash_config& c) { return c.kv_terms == 2 ? 2 : 1; }

size_t layer_pool_elems(const dflash_model_s* m, const dflash_kv* kv) {
  return static_cast<size_t>(kv->n_pages) * 2 * kv_terms_of(m->cfg) * m->cfg.n_kv_heads *
         m->cfg.page_size * m->cfg.head_dim;
}

void set_pool(const dflash_model_s* m, QkvEpi& e, const dflash_kv* kv, int layer) {
  if (kv->dtype == 1) {
    // E4M3 context cache: one byte per element, one scale per vector
    e.pool = nullptr;
    e.pool8 = static_cast<uint8_t*>(kv->pool) + layer_pool_elems(m, kv) * layer;
    e.scales8 = kv->scales + layer_pool_elems(m, kv) / m->cfg.head_dim * layer;
  } else {
    e.pool = static_cast<uint16_t*>(kv->pool) + layer_pool_elems(m, kv) * layer;
  }
  e.page_table = kv->page_table;
  e.max_pages = kv->max_pages;
  e.n_pages = kv->n_pages;
  e.n_req = kv->n_rows;
  e.kv_terms = kv_terms_of(m->cfg);
}

// Attention kernel of a stack pass over `batch` requests of n block rows.
// The drafter: all block rows per CTA, key splits from an occupancy model.
// The target (causal): query tiles of 64/G block rows and fixed 512-key
// splits, chosen per cache (never per call), so block verify and one-token
// decode run the same per-row arithmetic.
struct AttnPlan {
  bool use_tc;       // tcgen05 kernel (else mma.sync)
  int split_pages;   // pages per key split (tcgen05)
  int rows_per_tile; // block rows per query tile (tcgen05)
  int splits;        // key splits per (request, KV head) (tcgen05)
  uint64_t pool_rows;
};

AttnPlan attn_plan(const dflash_model_s* m, const dflash_kv* kv, int batch, int n) {
  const dflash_config& c = m->cfg;
  const int terms = kv_terms_of(c);
  const int G = c.n_q_heads / c.n_kv_heads;
  AttnPlan a;
  const int tc_pages = kv->max_pages + (m->is_draft ? (n + 15) / 16 : 0);
  a.split_pages = m->is_draft ? attention_tc_split_pages(c.head_dim, batch * c.n_kv_heads, tc_pages)
                              : attention_tc_target_split_pages();
  const int tc_splits = (tc_pages + a.split_pages - 1) / a.split_pages;
  a.splits = tc_splits;
  a.rows_per_tile = m->is_draft ? n : std::max(1, 64 / G);
  a.pool_rows = static_cast<uint64_t>(c.n_layers) * kv->n_pages * 2 * terms * c.n_kv_heads * 16;
  a.use_tc = m->attn_tc && a.pool_rows + 16 < (1ull << 31) &&
             (m->is_draft ? attention_tc_ok(c.head_dim, c.n_q_heads, c.n_kv_heads, n, c.page_size,
                                            a.split_pages)
                          : ((c.head_dim == 64 || c.head_dim == 128) && G <= 64 &&
                             tc_splits <= kMaxAttnCluster));
  return a;
}

int check_kv(const dflash_model_s* m, const dflash_kv* kv) {
  if (kv == nullptr || kv->pool == nullptr || kv->page_table == nullptr || kv->n_pages <= 0 ||
      kv->max_pages <= 0 || kv->n_rows <= 0 || (kv->dtype != 0 && kv->dtype != 1))
    return DFLASH_ERR_INVALID_ARG;
  if (!aligned16(kv->pool)) return DFLASH_ERR_INVALID_ARG;
  if (kv->dtype == 1) {
    // E4M3 caches: drafter context caches with one-term K/V only
    if (kv->scales == nullptr || !aligned16(kv->scales)) return DFLASH_ERR_INVALID_ARG;
    if (!m->is_draft || kv_terms_of(m->cfg) != 1) return DFLASH_ERR_UNSUPPORTED;
  }
  return DFLASH_OK;
}

void set_norm_in(const dflash_model_s* m, GemmParams& p, const float* ssq, int norm_rows) {
  p.ssq_in = ssq;
  p.ssq_in_tiles = m->cfg.hidden / kTileN;
  p.norm_rows = norm_rows;
  p.norm_dim = m->cfg.hidden;
  p.norm_eps = m->cfg.rms_eps;
}

void set_resid_out(const dflash_model_s* m, GemmParams& p, float* x, const uint16_t* gnext,
                   uint16_t* xg, float* ssq) {
  p.mode = EPI_RESID;
  p.resid = x;
  p.ld_resid = m->cfg.hidden;
  p.gnext = gnext;
  p.xg_out = xg;
  p.ld_xg = m->cfg.hidden;
  p.ssq_out = ssq;
  p.ssq_ld = m->cfg.hidden / kTileN;
}

// One decoder-layer stack pass.  On entry b.x holds the residual stream,
// b.a its first-norm input bf16(x * in_norm[0]) (+ context rows after the
// block rows for the drafter) and b.ssq_a the row sums of squares.  Every
// RMSNorm is folded into the GEMM epilogues (see GemmParams::ssq_in).
// On exit b.a2 / b.ssq_a2 hold the final-norm input for the LM head.
int run_stack(const dflash_model_s* m, Ws& ws, StackBufs& b, int batch, int n,
              const int32_t* pos0, const dflash_kv* kv, int ctx_rows, const int32_t* ctx_req,
              const int32_t* ctx_pos, const int32_t* tap_slot, int n_taps, uint16_t* taps,
              cudaStream_t s) {
  const dflash_config& c = m->cfg;
  const int rows = batch * n;
  const int H = c.hidden;
  const int max_keys = kv->max_pages * c.page_size;
  // attention on tcgen05: tensor maps over the pool and the block K/V
  const int terms = kv_terms_of(c);
  const AttnPlan plan = attn_plan(m, kv, batch, n);
  const int tc_split_pages = plan.split_pages;
  const int tc_rows_per_tile = plan.rows_per_tile;
  const uint64_t pool_rows = plan.pool_rows;
  const bool use_tc = plan.use_tc;
  const int tc_splits = plan.splits;
  const bool fp8 = kv->dtype == 1;
  if (fp8 && !use_tc) return DFLASH_ERR_UNSUPPORTED;  // E4M3 caches: tcgen05 attention only
  // K pages as 2-D boxes (one per 64-column half), V pages as 3-D boxes
  // (both halves of a page in one box); E4M3 pools: one uint8 map of codes
  CUtensorMap pool_map, pool_v_map, kblk_map, vblk_map;
  if (use_tc) {
    int rc = fp8 ? encode_map_u8(&pool_map, kv->pool, pool_rows, c.head_dim, 16)
                 : encode_map(&pool_map, kv->pool, pool_rows, c.head_dim, c.head_dim, 16);
    if (!rc)
      rc = encode_map(&kblk_map, b.kblk, static_cast<uint64_t>(rows) * c.n_kv_heads, c.head_dim,
                      c.head_dim, 16);
    if (!rc)
      rc = encode_map_rows16(&vblk_map, b.vblk, static_cast<uint64_t>(rows) * c.n_kv_heads,
                             c.head_dim);
    if (!rc) {
      if (fp8)
        pool_v_map = vblk_map;  // unused: the E4M3 kernel reads V codes through pool_map
      else
        rc = encode_map_rows16(&pool_v_map, kv->pool, pool_rows, c.head_dim);
    }
    if (rc) return rc;
  }
  // Two-term (hi + lo bf16) activations for O, gate/up and down.  The
  // target: every layer, for any row count (its per-row arithmetic must not
  // depend on the batch).  The drafter: every layer while the pass has at
  // most 64 block rows (its GEMMs then stream weights and the second term
  // is free), else the first two layers, which carry most of the rounding
  // error that reaches the logits.
  const int two_layers = m->two_term_layers >= 0 ? m->two_term_layers
                         : (m->is_draft && rows > 64) ? std::min(2, c.n_layers)
                                                      : c.n_layers;
  for (int l = 0; l < c.n_layers; ++l) {
    const bool two = l < two_layers;  // hi + lo activations in this layer
    // QKV (+ context K/V rows in the same weight pass)
    {
      const int M = rows + ctx_rows;
      GemmParams p = gemm_base(m, M, m->qkv_rows, H, gemm_bn_for(M, m->qkv_rows, m->sms), ws);
      p.w_row0 = l * m->qkv_rows;
      p.mode = EPI_QKV;
      set_norm_in(m, p, b.ssq_a, rows);
      QkvEpi e = qkv_base(m, l);
      set_pool(m, e, kv, l);
      e.q = b.q;
      if (m->is_draft) {
        e.n_blk = rows;
        e.block = n;
        e.anchor_pos = pos0;
        e.pool_req = ctx_req;
        e.pool_pos = ctx_pos;
        e.keep_q_pool = 0;
        e.kblk = b.kblk;
        e.vblk = b.vblk;
      } else {
        e.n_blk = 0;
        e.rows_per_req = n;
        e.pool_pos0 = pos0;
        e.keep_q_pool = 1;
      }
      p.qkv = e;
      int rc = run_gemm(m, &m->m_wqkv, b.a, H, p, b.partial, s);
      if (rc) return rc;
    }
    // attention
    if (use_tc) {
      AttnTcParams a;
      std::memset(&a, 0, sizeof(a));
      a.q = b.q;
      a.batch = batch;
      a.n = n;
      a.pos0 = pos0;
      a.page_table = kv->page_table;
      a.max_pages = kv->max_pages;
      a.n_pages = kv->n_pages;
      a.hq = c.n_q_heads;
      a.hkv = c.n_kv_heads;
      a.d = c.head_dim;
      a.pool_row0 = static_cast<int>(static_cast<uint64_t>(l) * kv->n_pages * 2 * terms *
                                     c.n_kv_heads * 16);
      a.pool_rows = static_cast<int>(pool_rows);
      a.split_pages = tc_split_pages;
      a.n_splits = tc_splits;
      a.rows_per_tile = tc_rows_per_tile;
      a.causal = m->is_draft ? 0 : 1;
      a.kv_terms = terms;
      a.fp8 = fp8 ? 1 : 0;
      a.scales = kv->scales;
      a.out = b.o;
      a.out_lo = two ? b.o_lo : nullptr;
      a.status = ws.status();
      DF_CUDA(attention_tc_launch(&pool_map, &pool_v_map, &kblk_map, &vblk_map, a, s, true));
    } else {
      AttnParams a;
      std::memset(&a, 0, sizeof(a));
      a.q = b.q;
      a.batch = batch;
      a.n = n;
      a.pos0 = pos0;
      a.causal = m->is_draft ? 0 : 1;
      a.pool = static_cast<const uint16_t*>(kv->pool) + layer_pool_elems(m, kv) * l;
      a.kv_terms = kv_terms_of(c);
      a.page_table = kv->page_table;
      a.max_pages = kv->max_pages;
      a.n_pages = kv->n_pages;
      a.page_size = c.page_size;
      a.kblk = b.kblk;
      a.vblk = b.vblk;
      a.hq = c.n_q_heads;
      a.hkv = c.n_kv_heads;
      a.d = c.head_dim;
      a.split_keys = attn_split_keys(m, batch, max_keys);
      a.n_splits = attn_n_splits(m, a.split_keys, max_keys);
      a.cluster = attention_cluster_ok(c.head_dim, c.n_q_heads, c.n_kv_heads, a.n_splits) ? 1 : 0;
      a.o_part = b.o_part;
      a.ml_part = b.ml_part;
      a.out = b.o;
      a.out_lo = two ? b.o_lo : nullptr;
      a.status = ws.status();
      DF_CUDA(attention_launch(a, s, true));
    }
    // O projection + residual (+ DFlash-2 block conv) -> post-norm input
    {
      GemmParams p = gemm_base(m, rows, H, m->q_dim, gemm_bn_for(rows, H, m->sms), ws);
      p.w_row0 = l * H;
      set_resid_out(m, p, b.x, u16(m->w.post_norm) + static_cast<size_t>(l) * H, b.a2, b.ssq_a2);
      p.xg_lo = two ? b.a2_lo : nullptr;
      if (m->is_draft && c.conv_width > 0 && m->w.conv != nullptr) {
        p.conv = u16(m->w.conv) + static_cast<size_t>(l) * H * c.conv_width;
        p.conv_width = c.conv_width;
        p.block = n;
      }
      int rc = run_gemm(m, &m->m_wo, b.o, m->q_dim, p, b.partial, s, two ? b.o_lo : nullptr);
      if (rc) return rc;
    }
    // gate/up + SwiGLU: each 128-row tile = 64 gate rows + the matching 64 up rows
    {
      GemmParams p = gemm_base(m, rows, 2 * c.mlp, H, gemm_bn_for(rows, 2 * c.mlp, m->sms), ws);
      p.w_row0 = l * 2 * c.mlp;
      p.w_tile_step = 64;
      p.w_half_gap = c.mlp;
      p.mode = EPI_SWIGLU;
      p.out = b.hmid;
      p.out_lo = two ? b.hmid_lo : nullptr;
      p.ld_out = c.mlp;
      set_norm_in(m, p, b.ssq_a2, rows);
      int rc = run_gemm(m, &m->m_gu, b.a2, H, p, b.partial, s, two ? b.a2_lo : nullptr);
      if (rc) return rc;
    }
    // down projection + residual -> next layer's in-norm input (or final norm)
    {
      GemmParams p = gemm_base(m, rows, H, c.mlp, gemm_bn_for(rows, H, m->sms), ws);
      p.w_row0 = l * H;
      const bool last = (l == c.n_layers - 1);
      const uint16_t* g = last ? u16(m->w.final_norm)
                               : u16(m->w.in_norm) + static_cast<size_t>(l + 1) * H;
      set_resid_out(m, p, b.x, g, last ? b.a2 : b.a, last ? b.ssq_a2 : b.ssq_a);
      if (taps != nullptr && tap_slot[l] >= 0) {
        p.raw_out = taps + static_cast<size_t>(tap_slot[l]) * H;
        p.ld_raw = n_taps * H;
      }
      int rc = run_gemm(m, &m->m_down, b.hmid, c.mlp, p, b.partial, s, two ? b.hmid_lo : nullptr);
      if (rc) return rc;
    }
  }
  return DFLASH_OK;
}

int run_lm_head(const dflash_model_s* m, Ws& ws, StackBufs& b, int rows, int block,
                int skip_first, int32_t* out, float* logits, cudaStream_t s) {
  const dflash_config& c = m->cfg;
  GemmParams p = gemm_base(m, rows, c.vocab, c.hidden, gemm_bn_for(rows, c.vocab, m->sms), ws);
  p.mode = EPI_ARGMAX;
  p.amax_val = b.amax_val;
  p.amax_idx = b.amax_idx;
  p.logits = logits;
  p.ld_logits = c.vocab;
  if (b.ssq_a2 != nullptr) set_norm_in(m, p, b.ssq_a2, rows);
  p.splits = 1;  // argmax needs the full dot product per tile
  p.kb_per_split = p.kb_total;
  const bool fused = rows <= kMaxAmaxKeyRows;
  if (fused) {
    // the cross-tile argmax finishes inside the GEMM launch
    p.amax_key = ws.amax_keys();
    p.amax_ticket = ws.status() + 2;
    p.amax_out = out;
    p.amax_block = block;
    p.amax_skip_first = skip_first;
  }
  int rc = run_gemm(m, &m->m_lm, b.a2, c.hidden, p, b.partial, s);
  if (rc) return rc;
  if (!fused)
    DF_CUDA(argmax_reduce_launch(b.amax_val, b.amax_idx, rows, c.vocab / kTileN, block, out,
                                 skip_first, s, true));
  return DFLASH_OK;
}

int check_cfg(const dflash_config* c, bool draft) {
  // hidden <= 8192: the row kernels hold a row in registers (8 columns x 4
  // chunks per thread of 256)
  if (c->n_layers < 1 || c->hidden < 128 || c->hidden % 128 || c->hidden > 8192 ||
      c->vocab < 128 || c->vocab % 128)
    return DFLASH_ERR_UNSUPPORTED;
  if (c->head_dim != 64 && c->head_dim != 128) return DFLASH_ERR_UNSUPPORTED;
  if (c->n_kv_heads < 1 || c->n_q_heads % c->n_kv_heads) return DFLASH_ERR_UNSUPPORTED;
  const int g = c->n_q_heads / c->n_kv_heads;
  if (g != 1 && g != 2 && g != 4 && g != 8) return DFLASH_ERR_UNSUPPORTED;
  if (((c->n_q_heads + 2 * c->n_kv_heads) * c->head_dim) % 128) return DFLASH_ERR_UNSUPPORTED;
  if ((c->n_q_heads * c->head_dim) % 64 || c->mlp < 64 || c->mlp % 64) return DFLASH_ERR_UNSUPPORTED;
  if (c->page_size != 16) return DFLASH_ERR_UNSUPPORTED;
  if (c->kv_terms < 0 || c->kv_terms > 2 || (draft && c->kv_terms == 2)) return DFLASH_ERR_UNSUPPORTED;
  if (draft) {
    if (c->block < 1 || c->block > 32 || 256 % c->block) return DFLASH_ERR_UNSUPPORTED;
    if (c->n_taps < 1) return DFLASH_ERR_UNSUPPORTED;
    if (c->conv_width < 0 || c->conv_width > 7 || (c->conv_width && c->conv_width % 2 == 0))
      return DFLASH_ERR_UNSUPPORTED;
  }
  if (!(c->rms_eps >= 0.f) || !(c->rope_base > 1.f)) return DFLASH_ERR_INVALID_ARG;
  return DFLASH_OK;
}

}  // namespace

namespace dflash {
// Argument and capacity checks of dflash_ctx_fuse (nothing is launched).
int ctx_fuse_check(const dflash_model_s* m, const void* taps, int32_t T, const void* ctx,
                   const void* ws, size_t ws_bytes) {
  if (m == nullptr || !m->is_draft || taps == nullptr || ctx == nullptr || ws == nullptr || T < 1)
    return DFLASH_ERR_INVALID_ARG;
  if (!aligned16(taps) || !aligned16(ctx) || (reinterpret_cast<uintptr_t>(ws) & 255))
    return DFLASH_ERR_INVALID_ARG;
  Ws w;
  w.dry = true;
  w.take<float>(partial_floats(m, 0, T));
  w.take<float>(static_cast<size_t>(T) * m->cfg.hidden);
  return w.off > ws_bytes ? DFLASH_ERR_CAPACITY : DFLASH_OK;
}
}  // namespace dflash

// ======================================================================= ABI
extern "C" {

const char* dflash_strerror(int code) {
  switch (code) {
    case DFLASH_OK: return "ok";
    case DFLASH_ERR_INVALID_ARG: return "invalid argument";
    case DFLASH_ERR_UNSUPPORTED: return "unsupported shape";
    case DFLASH_ERR_CAPACITY: return "capacity exceeded (workspace, page table or cache)";
    case DFLASH_ERR_CUDA: return "CUDA error";
    case DFLASH_ERR_TIMEOUT: return "device wait timed out";
    case DFLASH_ERR_NO_DEVICE: return "no compute-capability 10.3 device or driver entry point";
    default: return "unknown error";
  }
}

int dflash_last_cuda_error(void) { return g_last_cuda; }

uint64_t dflash_kernel_launches(void) { return dflash::launch_count(); }

int dflash_model_create(const dflash_config* cfg, const dflash_weights* w, dflash_model* out) {
  if (cfg == nullptr || w == nullptr || out == nullptr) return DFLASH_ERR_INVALID_ARG;
  *out = nullptr;
  const bool draft = cfg->block > 0;
  int rc = check_cfg(cfg, draft);
  if (rc) return rc;
  const void* need[] = {w->embed, w->lm_head, w->final_norm, w->in_norm, w->wqkv, w->wo,
                        w->post_norm, w->w_gate_up, w->w_down};
  for (const void* p : need)
    if (p == nullptr || !aligned16(p)) return DFLASH_ERR_INVALID_ARG;
  if (cfg->qk_norm && (w->q_norm == nullptr || w->k_norm == nullptr)) return DFLASH_ERR_INVALID_ARG;
  if (draft && (w->fc == nullptr || w->mask_embed == nullptr || !aligned16(w->fc) ||
                !aligned16(w->mask_embed) ||
                (cfg->fc_norm && (w->fc_norm == nullptr || !aligned16(w->fc_norm)))))
    return DFLASH_ERR_INVALID_ARG;
  if (draft && cfg->conv_width > 0 && w->conv == nullptr) return DFLASH_ERR_INVALID_ARG;

  int dev = 0;
  DF_CUDA(cudaGetDevice(&dev));
  cudaDeviceProp prop;
  DF_CUDA(cudaGetDeviceProperties(&prop, dev));
  if (prop.major != 10 || prop.minor != 3) return DFLASH_ERR_NO_DEVICE;
  rc = load_encode();
  if (rc) return rc;

  dflash_model_s* m = new (std::nothrow) dflash_model_s();
  if (m == nullptr) return DFLASH_ERR_CAPACITY;
  m->cfg = *cfg;
  m->w = *w;
  m->device = dev;
  m->sms = prop.multiProcessorCount;
  m->is_draft = draft;
  {
    // DFLASH_ATTN_TC=0 keeps the drafter on the mma.sync attention kernel
    const char* t = std::getenv("DFLASH_ATTN_TC");
    m->attn_tc = !(t != nullptr && t[0] == '0');
    // DFLASH_TWO_TERM_LAYERS=k: two-term activations in the first k layers only
    const char* tt = std::getenv("DFLASH_TWO_TERM_LAYERS");
    if (tt != nullptr && tt[0] != '\0')
      m->two_term_layers = std::max(0, std::min(m->cfg.n_layers, std::atoi(tt)));
    // DFLASH_DEP_LEAD=k: a GEMM lets the next kernel launch when its producer
    // has k weight k-blocks left to request (-1: at the start)
    const char* dl = std::getenv("DFLASH_DEP_LEAD");
    if (dl != nullptr && dl[0] != 0) m->dep_lead = std::atoi(dl);
    const char* pm = std::getenv("DFLASH_PRE_MASK");
    if (pm != nullptr && pm[0] != 0) m->pre_mask = std::atoi(pm);
  }
  if (draft && m->attn_tc && (cfg->head_dim == 64 || cfg->head_dim == 128))
    attention_tc_prepare(cfg->head_dim);
  m->q_dim = cfg->n_q_heads * cfg->head_dim;
  m->kv_dim = cfg->n_kv_heads * cfg->head_dim;
  m->qkv_rows = m->q_dim + 2 * m->kv_dim;
  const uint64_t L = cfg->n_layers, H = cfg->hidden, F = cfg->mlp;
  rc = encode_map(&m->m_wqkv, w->wqkv, L * m->qkv_rows, H, H, 64);
  if (!rc) rc = encode_map(&m->m_wo, w->wo, L * H, m->q_dim, m->q_dim, 64);
  if (!rc) rc = encode_map(&m->m_gu, w->w_gate_up, L * 2 * F, H, H, 64);
  if (!rc) rc = encode_map(&m->m_down, w->w_down, L * H, F, F, 64);
  if (!rc) rc = encode_map(&m->m_lm, w->lm_head, cfg->vocab, H, H, 64);
  if (!rc && draft)
    rc = encode_map(&m->m_fc, w->fc, H, static_cast<uint64_t>(cfg->n_taps) * H,
                    static_cast<uint64_t>(cfg->n_taps) * H, 64);
  if (rc) {
    delete m;
    return rc;
  }
  // inv_freq_p = base^(-2p/d) as an unevaluated (hi, lo) float pair
  const int half = cfg->head_dim / 2;
  for (int p = 0; p < kMaxRopePairs; ++p) {
    double f = p < half ? std::pow(static_cast<double>(cfg->rope_base),
                                   -2.0 * p / static_cast<double>(cfg->head_dim))
                        : 0.0;
    const float hi = static_cast<float>(f);
    m->rope[p] = make_float2(hi, static_cast<float>(f - static_cast<double>(hi)));
  }
  *out = m;
  return DFLASH_OK;
}

int dflash_model_destroy(dflash_model m) {
  delete m;
  return DFLASH_OK;
}

size_t dflash_workspace_bytes(dflash_model m, int32_t max_block_rows, int32_t max_ctx_rows,
                              int32_t max_batch, int32_t max_ctx_len) {
  if (m == nullptr || max_block_rows < 0 || max_ctx_rows < 0 || max_batch < 1 || max_ctx_len < 0)
    return 0;
  const dflash_config& c = m->cfg;
  const int max_keys = ((max_ctx_len + c.page_size - 1) / c.page_size) * c.page_size;
  size_t need = kHeaderBytes;
  // stack pass (draft block or target rows); block rows are batch*B, split across
  // the batch as n = rows / batch
  if (max_block_rows > 0) {
    Ws ws;
    ws.dry = true;
    StackBufs b;
    const int n = std::max(1, max_block_rows / max_batch);
    layout_stack(m, ws, b, max_batch, n, max_ctx_rows, max_keys);
    // the attention partials are sized for the worst split count over batch sizes
    for (int bt = 1; bt <= max_batch; bt *= 2) {
      const int nb = std::max(1, max_block_rows / bt);
      Ws w2;
      w2.dry = true;
      StackBufs b2;
      layout_stack(m, w2, b2, bt, nb, max_ctx_rows, max_keys);
      need = std::max(need, w2.off);
    }
    need = std::max(need, ws.off);
  }
  if (max_ctx_rows > 0 && m->is_draft) {
    Ws ws;
    ws.dry = true;
    ws.take<float>(partial_floats(m, 0, max_ctx_rows));
    ws.take<float>(static_cast<size_t>(max_ctx_rows) * c.hidden);
    need = std::max(need, ws.off);
  }
  return need;
}

int dflash_workspace_init(void* ws, size_t ws_bytes, void* stream) {
  if (ws == nullptr || ws_bytes < kHeaderBytes || (reinterpret_cast<uintptr_t>(ws) & 255))
    return DFLASH_ERR_INVALID_ARG;
  DF_CUDA(cudaMemsetAsync(ws, 0, kHeaderBytes, static_cast<cudaStream_t>(stream)));
  return DFLASH_OK;
}

int dflash_get_status(const void* ws, int32_t* status, int32_t* site, void* stream) {
  if (ws == nullptr || status == nullptr) return DFLASH_ERR_INVALID_ARG;
  int32_t h[2] = {0, 0};
  DF_CUDA(cudaStreamSynchronize(static_cast<cudaStream_t>(stream)));
  DF_CUDA(cudaMemcpy(h, ws, sizeof(h), cudaMemcpyDeviceToHost));
  *status = h[0];
  if (site) *site = h[1];
  return DFLASH_OK;
}

int dflash_ctx_fuse(dflash_model m, const void* taps, int32_t T, void* ctx, void* ws,
                    size_t ws_bytes, void* stream) {
  int rc = dflash::ctx_fuse_check(m, taps, T, ctx, ws, ws_bytes);
  if (rc) return rc;
  const dflash_config& c = m->cfg;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Ws w;
  w.base = static_cast<uint8_t*>(ws);
  float* partial = w.take<float>(partial_floats(m, 0, T));
  float* cf = w.take<float>(static_cast<size_t>(T) * c.hidden);
  const int K = c.n_taps * c.hidden;
  GemmParams p = gemm_base(m, T, c.hidden, K, gemm_bn_for(T, c.hidden, m->sms), w);
  if (c.fc_norm) {
    p.mode = EPI_STORE_F32;
    p.out = cf;
  } else {
    p.mode = EPI_STORE_BF16;
    p.out = ctx;
  }
  p.ld_out = c.hidden;
  rc = run_gemm(m, &m->m_fc, taps, K, p, partial, s);
  if (rc) return rc;
  if (c.fc_norm)
    DF_CUDA(rmsnorm_launch(cf, T, c.hidden, u16(m->w.fc_norm), c.rms_eps,
                           static_cast<uint16_t*>(ctx), c.hidden, nullptr, 0, s, true));
  return DFLASH_OK;
}

int dflash_kv_append(dflash_model m, const void* ctx, const int32_t* row_req,
                     const int32_t* row_pos, int32_t T, const dflash_kv* kv, void* ws,
                     size_t ws_bytes, void* stream) {
  if (m == nullptr || !m->is_draft || ctx == nullptr || row_req == nullptr ||
      row_pos == nullptr || T < 1 || ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255) ||
      !aligned16(ctx))
    return DFLASH_ERR_INVALID_ARG;
  int rc = check_kv(m, kv);
  if (rc) return rc;
  const dflash_config& c = m->cfg;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Ws w;
  w.base = static_cast<uint8_t*>(ws);
  float* partial = w.take<float>(partial_floats(m, 0, T));
  if (w.off > ws_bytes) return DFLASH_ERR_CAPACITY;
  for (int l = 0; l < c.n_layers; ++l) {
    GemmParams p = gemm_base(m, T, 2 * m->kv_dim, c.hidden, gemm_bn_for(T, 2 * m->kv_dim, m->sms), w);
    p.w_row0 = l * m->qkv_rows + m->q_dim;
    p.mode = EPI_QKV;
    QkvEpi e = qkv_base(m, l);
    set_pool(m, e, kv, l);
    e.n_blk = 0;
    e.pool_req = row_req;
    e.pool_pos = row_pos;
    e.keep_q_pool = 0;
    e.f0 = m->q_dim;
    p.qkv = e;
    rc = run_gemm(m, &m->m_wqkv, ctx, c.hidden, p, partial, s);
    if (rc) return rc;
  }
  return DFLASH_OK;
}

int dflash_draft_block(dflash_model m, const int32_t* anchor, const int32_t* anchor_pos,
                       int32_t batch, const dflash_kv* kv, const void* pending_ctx,
                       const int32_t* pending_req, const int32_t* pending_pos, int32_t T,
                       int32_t* draft, float* logits, float* hidden, void* ws, size_t ws_bytes,
                       void* stream) {
  if (m == nullptr || !m->is_draft || anchor == nullptr || anchor_pos == nullptr || batch < 1 ||
      draft == nullptr || ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255) || T < 0)
    return DFLASH_ERR_INVALID_ARG;
  if (T > 0 && (pending_ctx == nullptr || pending_req == nullptr || pending_pos == nullptr ||
                !aligned16(pending_ctx)))
    return DFLASH_ERR_INVALID_ARG;
  int rc = check_kv(m, kv);
  if (rc) return rc;
  if (batch > kv->n_rows) return DFLASH_ERR_CAPACITY;
  // E4M3 caches: tcgen05 attention only (refused before anything launches)
  if (kv->dtype == 1 && !attn_plan(m, kv, batch, m->cfg.block).use_tc)
    return DFLASH_ERR_UNSUPPORTED;
  const dflash_config& c = m->cfg;
  const int B = c.block;
  const int rows = batch * B;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Ws w;
  w.base = static_cast<uint8_t*>(ws);
  StackBufs b;
  const int max_keys = kv->max_pages * c.page_size;
  layout_stack(m, w, b, batch, B, T, max_keys);
  if (w.off > ws_bytes) return DFLASH_ERR_CAPACITY;
  DF_CUDA(embed_block_launch(anchor, batch, B, u16(m->w.embed), u16(m->w.mask_embed),
                             u16(m->w.in_norm), c.hidden, b.x, b.a, c.hidden, b.ssq_a,
                             u16(pending_ctx), T, s, true, w.status(), c.vocab));
  rc = run_stack(m, w, b, batch, B, anchor_pos, kv, T, pending_req, pending_pos, nullptr, 0,
                 nullptr, s);
  if (rc) return rc;
  if (B > 1 || logits != nullptr) {
    rc = run_lm_head(m, w, b, rows, B, 1, draft, logits, s);
    if (rc) return rc;
  }
  if (hidden != nullptr)
    DF_CUDA(copy_rows_f32_launch(b.x, hidden, static_cast<size_t>(rows) * c.hidden, s, true));
  return DFLASH_OK;
}

int dflash_lm_head_argmax(dflash_model m, const void* x, int32_t rows, int32_t* argmax,
                          float* logits, void* ws, size_t ws_bytes, void* stream) {
  if (m == nullptr || x == nullptr || rows < 1 || argmax == nullptr || ws == nullptr ||
      (reinterpret_cast<uintptr_t>(ws) & 255) || !aligned16(x))
    return DFLASH_ERR_INVALID_ARG;
  const dflash_config& c = m->cfg;
  Ws w;
  w.base = static_cast<uint8_t*>(ws);
  StackBufs b;
  std::memset(&b, 0, sizeof(b));
  const int vt = c.vocab / kTileN;
  b.amax_val = w.take<float>(static_cast<size_t>(rows) * vt);
  b.amax_idx = w.take<int32_t>(static_cast<size_t>(rows) * vt);
  if (w.off > ws_bytes) return DFLASH_ERR_CAPACITY;
  b.a2 = static_cast<uint16_t*>(const_cast<void*>(x));
  return run_lm_head(m, w, b, rows, 1, 0, argmax, logits, static_cast<cudaStream_t>(stream));
}

int dflash_verify_greedy(const int32_t* draft, const int32_t* target, int32_t batch, int32_t B,
                         int32_t* out_tokens, int32_t* n_accept, const int32_t* tgt_len_in,
                         int32_t* tgt_len_out, int32_t* ctx_pending, int32_t* anchor_out,
                         const int32_t* anchor_pos_in, int32_t* anchor_pos_out, int32_t* ctx_pos,
                         void* stream) {
  if (target == nullptr || batch < 1 || B < 1 || B > 32 || (B > 1 && draft == nullptr))
    return DFLASH_ERR_INVALID_ARG;
  if ((tgt_len_out != nullptr && tgt_len_in == nullptr) ||
      ((anchor_pos_out != nullptr || ctx_pos != nullptr) && anchor_pos_in == nullptr))
    return DFLASH_ERR_INVALID_ARG;
  DF_CUDA(verify_launch(draft, target, batch, B, out_tokens, n_accept, tgt_len_in, tgt_len_out,
                        ctx_pending, anchor_out, anchor_pos_in, anchor_pos_out, ctx_pos,
                        static_cast<cudaStream_t>(stream), true));
  return DFLASH_OK;
}

int dflash_kv_quantize(dflash_model m, const dflash_kv* src, const dflash_kv* dst, void* stream) {
  if (m == nullptr || src == nullptr || dst == nullptr || src->pool == nullptr ||
      dst->pool == nullptr || dst->scales == nullptr || src->dtype != 0 || dst->dtype != 1 ||
      src->n_pages != dst->n_pages || src->n_pages <= 0)
    return DFLASH_ERR_INVALID_ARG;
  if (!aligned16(src->pool) || !aligned16(dst->pool) || !aligned16(dst->scales))
    return DFLASH_ERR_INVALID_ARG;
  const dflash_config& c = m->cfg;
  if (kv_terms_of(c) != 1) return DFLASH_ERR_UNSUPPORTED;
  const size_t vectors = static_cast<size_t>(c.n_layers) * src->n_pages * 2 * c.n_kv_heads *
                         c.page_size;
  DF_CUDA(kv_quantize_launch(static_cast<const uint16_t*>(src->pool),
                             static_cast<uint8_t*>(dst->pool), dst->scales, vectors, c.head_dim,
                             static_cast<cudaStream_t>(stream), true));
  return DFLASH_OK;
}

size_t dflash_sampling_workspace_bytes(int32_t batch, int32_t B) {
  if (batch < 1 || B < 1) return 0;
  return kHeaderBytes + al256(static_cast<size_t>(batch) * (2 * B - 1) * sizeof(double2));
}

int dflash_verify_sampling(const int32_t* draft, const float* draft_logits,
                           const float* target_logits, int32_t batch, int32_t B, int32_t vocab,
                           double temperature, const double* u, const double* w,
                           int32_t* out_tokens, int32_t* n_accept, const int32_t* tgt_len_in,
                           int32_t* tgt_len_out, int32_t* ctx_pending, int32_t* anchor_out,
                           const int32_t* anchor_pos_in, int32_t* anchor_pos_out, int32_t* ctx_pos,
                           void* ws, size_t ws_bytes, void* stream) {
  if (target_logits == nullptr || w == nullptr || out_tokens == nullptr || batch < 1 || B < 1 ||
      B > 32 || vocab < 1 || !(temperature > 0.0) || !std::isfinite(temperature))
    return DFLASH_ERR_INVALID_ARG;
  if (B > 1 && (draft == nullptr || draft_logits == nullptr || u == nullptr))
    return DFLASH_ERR_INVALID_ARG;
  if ((tgt_len_out != nullptr && tgt_len_in == nullptr) ||
      ((anchor_pos_out != nullptr || ctx_pos != nullptr) && anchor_pos_in == nullptr))
    return DFLASH_ERR_INVALID_ARG;
  if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255)) return DFLASH_ERR_INVALID_ARG;
  if (ws_bytes < dflash_sampling_workspace_bytes(batch, B)) return DFLASH_ERR_CAPACITY;
  uint8_t* base = static_cast<uint8_t*>(ws);
  DF_CUDA(verify_sampling_launch(draft, draft_logits, target_logits, batch, B, vocab, temperature,
                                 u, w, reinterpret_cast<double2*>(base + kHeaderBytes), out_tokens,
                                 n_accept, tgt_len_in, tgt_len_out, ctx_pending, anchor_out,
                                 anchor_pos_in, anchor_pos_out, ctx_pos,
                                 reinterpret_cast<int32_t*>(base),
                                 static_cast<cudaStream_t>(stream), true));
  return DFLASH_OK;
}

int dflash_sample_rows(const float* logits, int32_t n_blocks, int32_t block, int32_t skip_first,
                       int32_t vocab, double temperature, const double* a, int32_t* out,
                       void* ws, size_t ws_bytes, void* stream) {
  if (logits == nullptr || a == nullptr || out == nullptr || n_blocks < 1 || block < 1 ||
      (skip_first != 0 && skip_first != 1) || block - skip_first < 1 || vocab < 1 ||
      !(temperature > 0.0) || !std::isfinite(temperature))
    return DFLASH_ERR_INVALID_ARG;
  if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255)) return DFLASH_ERR_INVALID_ARG;
  const size_t used = static_cast<size_t>(n_blocks) * (block - skip_first);
  if (used > (1u << 30) || ws_bytes < kHeaderBytes + al256(used * sizeof(double2)))
    return DFLASH_ERR_CAPACITY;
  DF_CUDA(sample_rows_launch(logits, static_cast<int>(used), block, skip_first, vocab, temperature,
                             a, reinterpret_cast<double2*>(static_cast<uint8_t*>(ws) + kHeaderBytes),
                             out, static_cast<cudaStream_t>(stream), true));
  return DFLASH_OK;
}

int dflash_target_forward(dflash_model m, const int32_t* tokens, const int32_t* pos0,
                          int32_t batch, int32_t n, const dflash_kv* kv,
                          const int32_t* tap_layers, int32_t n_taps, void* taps,
                          int32_t* argmax, float* logits, void* ws, size_t ws_bytes,
                          void* stream) {
  if (m == nullptr || m->is_draft || tokens == nullptr || pos0 == nullptr || batch < 1 || n < 1 ||
      argmax == nullptr || ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255))
    return DFLASH_ERR_INVALID_ARG;
  if (n_taps < 0 || (n_taps > 0 && (tap_layers == nullptr || taps == nullptr)))
    return DFLASH_ERR_INVALID_ARG;
  int rc = check_kv(m, kv);
  if (rc) return rc;
  if (batch > kv->n_rows) return DFLASH_ERR_CAPACITY;
  const dflash_config& c = m->cfg;
  std::vector<int32_t> slot(c.n_layers, -1);
  for (int i = 0; i < n_taps; ++i) {
    if (tap_layers[i] < 0 || tap_layers[i] >= c.n_layers || slot[tap_layers[i]] >= 0)
      return DFLASH_ERR_INVALID_ARG;
    slot[tap_layers[i]] = i;
  }
  const int rows = batch * n;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Ws w;
  w.base = static_cast<uint8_t*>(ws);
  StackBufs b;
  layout_stack(m, w, b, batch, n, 0, kv->max_pages * c.page_size);
  if (w.off > ws_bytes) return DFLASH_ERR_CAPACITY;
  DF_CUDA(embed_tokens_launch(tokens, rows, u16(m->w.embed), u16(m->w.in_norm), c.hidden, b.x,
                              b.a, b.ssq_a, s, true, w.status(), c.vocab));
  rc = run_stack(m, w, b, batch, n, pos0, kv, 0, nullptr, nullptr, slot.data(), n_taps,
                 static_cast<uint16_t*>(taps), s);
  if (rc) return rc;
  return run_lm_head(m, w, b, rows, n, 0, argmax, logits, s);
}

int dflash_synth_target(const int32_t* draft, int32_t batch, int32_t B, const uint64_t* threshold,
                        int32_t vocab, uint64_t seed, int64_t* step, int32_t advance,
                        int32_t* target, void* stream) {
  if (threshold == nullptr || step == nullptr || target == nullptr || batch < 1 || B < 1 ||
      vocab < 2 || batch * B > 1024 || (B > 1 && draft == nullptr))
    return DFLASH_ERR_INVALID_ARG;
  DF_CUDA(synth_target_launch(draft, batch, B, threshold, vocab, seed, step, advance, target,
                              static_cast<cudaStream_t>(stream), true));
  return DFLASH_OK;
}

int dflash_selftest_wait(int32_t arrive, int64_t limit_ns, int64_t* waited_ns, void* ws,
                         size_t ws_bytes, void* stream) {
  if (ws == nullptr || ws_bytes < kHeaderBytes || (reinterpret_cast<uintptr_t>(ws) & 255) ||
      limit_ns < 1 || limit_ns > 1000000000LL ||
      (reinterpret_cast<uintptr_t>(waited_ns) & 7))
    return DFLASH_ERR_INVALID_ARG;
  DF_CUDA(wait_selftest_launch(arrive != 0, static_cast<uint64_t>(limit_ns),
                               static_cast<int*>(ws), waited_ns,
                               static_cast<cudaStream_t>(stream)));
  return DFLASH_OK;
}

}  // extern "C"
