// Internal launch interface between the C ABI (dflash_api.cu) and the kernels.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

struct dflash_model_s;

namespace dflash {

constexpr int kTileN = 128;      // weight rows per CTA tile (MMA M)
constexpr int kTileK = 64;       // K elements per pipeline stage (one 128-B swizzle row)
constexpr int kMaxRopePairs = 64;

// Argument and workspace-capacity checks of dflash_ctx_fuse; returns the
// DFLASH_* code the call would return before launching anything.
int ctx_fuse_check(const dflash_model_s* m, const void* taps, int32_t T, const void* ctx,
                   const void* ws, size_t ws_bytes);

// Host-side count of kernel launches issued by this library.
uint64_t launch_count();
void count_launch();

enum EpiMode : int {
  EPI_STORE_BF16 = 0,  // out[m][n] = bf16(acc)
  EPI_STORE_F32 = 1,   // out[m][n] = acc
  EPI_RESID = 2,       // resid[m][n] += acc, then optional block conv
  EPI_SWIGLU = 3,      // out[m][j] = bf16(silu(gate) * up)
  EPI_QKV = 4,         // q/k norm + RoPE, route to q / block K,V / paged pool
  EPI_ARGMAX = 5,      // per-tile (max, argmax) per row (+ optional f32 logits)
};

struct QkvEpi {
  int n_blk;             // rows [0, n_blk) are block rows: request m / block, position anchor_pos + m % block
  int block;
  const int32_t* anchor_pos;
  int rows_per_req;      // pool rows (m >= n_blk): request (m - n_blk) / rows_per_req ... when pool_req == null
  const int32_t* pool_pos0;   // [batch] first position of each request's pool rows (target rows)
  const int32_t* pool_req;    // [rows] explicit request of each pool row (context rows), or null
  const int32_t* pool_pos;    // [rows] explicit position (< 0 = skip), or null
  int keep_q_pool;       // pool rows also store q (target forward)
  int n_q_heads, n_kv_heads, head_dim;
  int f0;                // feature index (in q|k|v space) of this launch's output feature 0
  const uint16_t* q_norm;  // [d] or null
  const uint16_t* k_norm;  // [d] or null
  float eps;
  uint16_t* q;           // [rows][hq][d]
  uint16_t* kblk;        // [batch][hkv][block][d]
  uint16_t* vblk;
  uint16_t* pool;        // layer base [n_pages][2][hkv][page][d]
  const int32_t* page_table;
  int max_pages, n_pages, page_size;
  int n_req;             // rows of page_table: explicit pool_req values must lie in [0, n_req)
  int kv_terms;          // 1: bf16 K/V planes; 2: also bf16 low terms (planes 2, 3)
  uint8_t* pool8;        // E4M3 context cache (layer base) instead of pool, or null
  float* scales8;        // its per-vector scales (layer base)
  float2 rope[kMaxRopePairs];  // inv_freq of pair p as (hi, lo) float pair
};

struct GemmParams {
  int M, N, K;           // activation rows, output features (this launch), reduction
  int w_row0;            // tensor-map row of output tile 0, half 0
  int w_tile_step;       // tensor-map rows advanced per output tile
  int w_half_gap;        // tensor-map row distance between the two 64-row halves
  int kb_total, kb_per_split, splits;
  int cluster;           // splits > 1: 1 = reduce through a thread-block cluster (DSMEM), 0 = global
  float* partial;        // [splits][M][N] (splits > 1)
  int32_t* counters;     // [n_tiles * m_tiles], zero between launches
  int32_t* status;
  int mode;
  void* out;             // bf16/f32 store or SwiGLU output
  int ld_out;
  // Optional low halves of the bf16 outputs that feed the next GEMM: the
  // value v is stored as hi = bf16(v) plus lo = bf16(v - hi), and the consumer
  // GEMM multiplies both (two MMAs into one accumulator), so the activation
  // operand carries ~16 significant bits instead of 8.
  uint16_t* out_lo;      // SwiGLU: [M][ld_out] next to out
  uint16_t* xg_lo;       // EPI_RESID: [M][ld_xg] next to xg_out
  float* resid;
  int ld_resid;
  const uint16_t* conv;  // [N][conv_width] (this layer) or null
  int conv_width, block;
  float* logits;         // argmax mode: optional [M][ld_logits]
  int ld_logits;
  float* amax_val;       // [M][n_tiles]
  int32_t* amax_idx;
  // Argmax finished inside the LM-head launch (amax_key != null): every CTA
  // folds its per-row (max, lowest index) into amax_key[m] with a 64-bit
  // atomic max, and the CTA that takes the last ticket writes the tokens to
  // amax_out (rows i % amax_block == 0 skipped when amax_skip_first: row m
  // goes to (m / B) * (B - 1) + i - 1) and clears the keys and the ticket.
  unsigned long long* amax_key;  // [M], zero between launches
  int32_t* amax_ticket;          // zero between launches
  int32_t* amax_out;
  int amax_block, amax_skip_first;
  // Deferred RMSNorm of the input rows: rows m < norm_rows of the result are
  // scaled by 1/sqrt(sum_t ssq_in[m][t] / norm_dim + norm_eps) (the input
  // operand holds bf16(x * g), the producer wrote per-tile sums of x^2).
  const float* ssq_in;
  int ssq_in_tiles, norm_rows, norm_dim;
  float norm_eps;
  // EPI_RESID outputs for the next norm: xg_out[m][n] = bf16(x_new * gnext[n]),
  // ssq_out[m][tile] = sum over the tile of x_new^2, raw_out = bf16(x_new).
  const uint16_t* gnext;
  uint16_t* xg_out;
  int ld_xg;
  float* ssq_out;
  int ssq_ld;
  uint16_t* raw_out;
  int ld_raw;
  QkvEpi qkv;
  int dep_lead;          // < 0: signal dependents at the start; else with dep_lead k-blocks left to load
  int pre_mask;          // epilogue inputs loaded during the main loop: 1 row scales, 2 QKV
                         // routing, 4 residual rows, 8 QKV gains and RoPE tables
};

// MMA N width (activation rows per tile) for M rows and N output features
// on a device with `sms` SMs.
int gemm_bn_for(int M, int N, int sms);
int gemm_max_smem_bytes();
// Clusters of `cluster` CTAs (BN variant) that can be resident at once.
int gemm_max_active_clusters(int bn, int cluster);
// x_lo_map (nullable): the low halves of a split activation operand
// (same shape as x_map); when given, every k-step issues a second MMA on it.
cudaError_t gemm_launch(const CUtensorMap* w_map, const CUtensorMap* x_map,
                        const CUtensorMap* x_lo_map, const GemmParams& p, int bn, cudaStream_t s,
                        bool pdl);

struct AttnParams {
  const uint16_t* q;     // [batch*n][hq][d]
  int batch, n;          // requests, query rows per request
  const int32_t* pos0;   // [batch] position of each request's row 0
  int causal;            // 1: row at pos attends keys [0, pos] of the pool; 0: [0, pos0) + block keys
  const uint16_t* pool;  // layer base
  const int32_t* page_table;
  int max_pages, n_pages, page_size;
  int kv_terms;          // 2: K and V also have bf16 low-term planes (2, 3)
  const uint16_t* kblk;  // [batch][hkv][n][d] (non-causal)
  const uint16_t* vblk;
  int hq, hkv, d;
  int split_keys;        // keys per split, multiple of 64
  int n_splits;          // grid.x
  int cluster;           // 1: the splits of a query tile form a cluster and combine through DSMEM
  float* o_part;         // [n_splits][batch*n][hq][d]
  float* ml_part;        // [n_splits][batch*n][hq][2]
  uint16_t* out;         // [batch*n][hq][d]
  uint16_t* out_lo;      // optional low halves bf16(o - bf16(o)) for the O-projection GEMM
  int32_t* status;
};
cudaError_t attention_launch(const AttnParams& p, cudaStream_t s, bool pdl);

// Attention on tcgen05 (attention_tc05.cu).  K/V come from three 2-D tensor
// maps: the whole pool viewed as [n_layers*n_pages*planes*hkv*16][d] rows
// (bf16: box 16 rows x 64 columns, 128-byte swizzle; E4M3 codes: uint8, box
// 16 rows x d bytes, no swizzle), and the block keys/values viewed as bf16
// [batch*hkv*n][d].
struct AttnTcParams {
  const uint16_t* q;     // [batch*n][hq][d]
  int batch, n;          // requests, block rows per request
  const int32_t* pos0;   // [batch] context length (keys [0, pos0) in the pool)
  const int32_t* page_table;
  int max_pages, n_pages;
  int hq, hkv, d;
  int pool_row0;         // pool-map row of this layer's page 0
  int pool_rows;         // rows of the pool map (a row index that reads as zeros)
  int split_pages;       // 16-key pages per key split
  int n_splits;          // key splits = cluster size (<= kMaxAttnCluster)
  int rows_per_tile;     // block rows per CTA (grid.z = query tiles); the drafter: n
  int causal;            // 1: target pass (pool keys [0, pos0 + i] for row i; no block keys)
  int kv_terms;          // 2: the pool pages hold K, V, K_lo, V_lo planes (causal only)
  int fp8;               // 1: pool_map is a uint8 map of E4M3 codes (box 16 rows x d bytes)
  const float* scales;   // E4M3: per-vector scales, indexed like the pool map's rows
  uint16_t* out;         // [batch*n][hq][d]
  uint16_t* out_lo;      // optional low halves
  int32_t* status;
};
// pool_map: 2-D, box 16 rows x 64 columns (bf16) or 16 rows x d bytes
// (E4M3 codes); pool_v_map, vblk_map: 3-D, box 16 rows x both column halves
// (pool_v_map unused by E4M3 caches); kblk_map: 2-D like pool_map.
cudaError_t attention_tc_launch(const CUtensorMap* pool_map, const CUtensorMap* pool_v_map,
                                const CUtensorMap* kblk_map, const CUtensorMap* vblk_map,
                                const AttnTcParams& p, cudaStream_t s, bool pdl);
// Pages per key split for `pairs` (request, KV head) pairs over
// `total_pages` 16-key pages (context pages + block pages).
int attention_tc_split_pages(int d, int pairs, int total_pages);
// Occupancy queries behind attention_tc_split_pages (call outside capture).
void attention_tc_prepare(int d);
// Key pages per split of the causal (target) variant: fixed.
int attention_tc_target_split_pages();
bool attention_tc_ok(int d, int hq, int hkv, int n, int page_size, int split_pages);
size_t attention_part_floats(int n_splits, int rows, int hq, int d);
bool attention_cluster_ok(int d, int hq, int hkv, int n_splits);
constexpr int kMaxAttnCluster = 16;

// small kernels (small_kernels.cu)
cudaError_t embed_block_launch(const int32_t* anchor, int batch, int block, const uint16_t* embed,
                               const uint16_t* mask_embed, const uint16_t* norm, int hidden,
                               float* x, uint16_t* a, int ld_a, float* ssq,
                               const uint16_t* pending, int T, cudaStream_t s, bool pdl,
                               int32_t* status, int vocab);
cudaError_t embed_tokens_launch(const int32_t* tokens, int rows, const uint16_t* embed,
                                const uint16_t* norm, int hidden, float* x, uint16_t* a,
                                float* ssq, cudaStream_t s, bool pdl, int32_t* status,
                                int vocab);
cudaError_t rmsnorm_launch(const float* x, int rows, int hidden, const uint16_t* g, float eps,
                           uint16_t* out, int ld_out, uint16_t* raw_out, int ld_raw,
                           cudaStream_t s, bool pdl);
cudaError_t argmax_reduce_launch(const float* val, const int32_t* idx, int rows, int n_tiles,
                                 int block, int32_t* out, int skip_first, cudaStream_t s,
                                 bool pdl);
cudaError_t verify_launch(const int32_t* draft, const int32_t* target, int batch, int B,
                          int32_t* out_tokens, int32_t* n_accept, const int32_t* tgt_len_in,
                          int32_t* tgt_len_out, int32_t* ctx_pending, int32_t* anchor_out,
                          const int32_t* anchor_pos_in, int32_t* anchor_pos_out, int32_t* ctx_pos,
                          cudaStream_t s, bool pdl);
cudaError_t synth_target_launch(const int32_t* draft, int batch, int B, const uint64_t* thr,
                                int vocab, uint64_t seed, int64_t* step, int advance,
                                int32_t* target, cudaStream_t s, bool pdl);
cudaError_t copy_rows_f32_launch(const float* src, float* dst, size_t n, cudaStream_t s, bool pdl);
// bf16 pool -> E4M3 codes + per-vector scales (vectors of d values)
cudaError_t kv_quantize_launch(const uint16_t* src, uint8_t* dst, float* scales, size_t vectors,
                               int d, cudaStream_t s, bool pdl);
// sampling.cu: verify at temperature T > 0 (stats: batch*(2B-1) double2), and
// categorical draws from softmax(logits / T) of the used rows of a blocked
// logits array (stats: n_used double2)
cudaError_t verify_sampling_launch(const int32_t* draft, const float* q_rows, const float* p_rows,
                                   int batch, int B, int V, double T, const double* u,
                                   const double* w, double2* stats, int32_t* out_tokens,
                                   int32_t* n_accept, const int32_t* tgt_len_in,
                                   int32_t* tgt_len_out, int32_t* ctx_pending,
                                   int32_t* anchor_out, const int32_t* anchor_pos_in,
                                   int32_t* anchor_pos_out, int32_t* ctx_pos, int32_t* status,
                                   cudaStream_t s, bool pdl);
cudaError_t sample_rows_launch(const float* rows, int n_used, int block, int skip, int V, double T,
                               const double* a, double2* stats, int32_t* out, cudaStream_t s,
                               bool pdl);
cudaError_t wait_selftest_launch(int arrive, uint64_t limit_ns, int* status, int64_t* waited_ns,
                                 cudaStream_t s);

}  // namespace dflash
