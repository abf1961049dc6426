// Weight-streaming GEMM on the 5th-generation tensor cores (tcgen05, sm_103a).
//
//   Y[m][n] = sum_k X[m][k] * W[n][k]        (y = x W^T, W stored [out][in])
//
// "Swap-AB" orientation: 128 weight rows form the MMA M side, the (few)
// activation rows the MMA N side (BN = 16..256), so a decode-sized batch
// still fills the 128-lane tensor core and the kernel streams W at HBM speed.
//
// Per CTA (128 threads): one 128-row weight tile x one BN-row activation tile
// over a K range (split-K).  Warp 0 lane 0 issues TMA loads into a STAGES-deep
// shared-memory ring (128-byte swizzle, 64 K-elements per stage); warp 1 owns
// the TMEM accumulator and lane 0 issues tcgen05.mma (M=128, N=BN, K=16, four
// per stage), committing each stage back to the producer through an mbarrier.
// With split-K, every CTA writes its fp32 partial tile and the last CTA of a
// tile (atomic ticket, no spinning) sums the partials in split order, so the
// result is deterministic and independent of M.  The final tile is staged in
// shared memory and handed to one of the fused epilogues (bf16/f32 store,
// residual add + DFlash-2 block conv, SwiGLU, q/k-norm + RoPE + KV routing,
// per-tile argmax for the LM head).
//
// Weight loads are issued before griddepcontrol.wait, so with programmatic
// dependent launch a GEMM prefetches its first stages of weights while the
// previous kernel is still draining.
#include "common.cuh"
#include "epilogue.cuh"
#include "kernels.h"

namespace dflash {

template <int BN, bool SPLIT>
struct GemmCfg {
  // BN <= 32 (decode-sized M): 3 CTAs fit per SM, so while a GEMM runs on two
  // slots the next kernel's CTAs (programmatic dependent launch) occupy the
  // third and prefetch their first weight stages.  A split activation operand
  // (hi + lo tiles) enlarges a stage, so those variants keep fewer stages.
  // (BN = 128: 3 stages of 32 KB, or 2 of 48 KB two-term, so two CTAs fit
  // per SM and each SM runs eight warps of epilogue)
  static constexpr int STAGES =
      SPLIT ? (BN <= 64 ? 3 : 2)
            : (BN <= 16 ? 4 : BN <= 32 ? 3 : BN <= 64 ? 4 : BN <= 128 ? 3 : 4);
  static constexpr int A_BYTES = kTileN * kTileK * 2;  // 16 KB
  static constexpr int B_BYTES = BN * kTileK * 2;      // one activation tile
  static constexpr int B_STAGE = SPLIT ? 2 * B_BYTES : B_BYTES;
  static constexpr int STAGE_BYTES = A_BYTES + B_STAGE;
  static constexpr int TS_LD = kTsLd;  // staged epilogue tile row stride (floats)
  static constexpr int TILE_BYTES = BN * TS_LD * 4;
  static constexpr int PIPE_BYTES = STAGES * STAGE_BYTES;
  static constexpr int MAIN_BYTES = PIPE_BYTES > TILE_BYTES ? PIPE_BYTES : TILE_BYTES;
  // epilogue scratch (row scales, QKV routing) sits after the staged tile;
  // before the epilogue the same place receives the split-K partials pushed
  // by the cluster peers ([splits][rows per CTA][128] fp32)
  static constexpr int SCRATCH_OFF = (TILE_BYTES + 255) / 256 * 256;
  static constexpr int RECV_OFF = SCRATCH_OFF;
  static_assert(SCRATCH_OFF + 4 * BN * 4 <= MAIN_BYTES, "epilogue scratch must fit the pipeline region");
  // Epilogue inputs loaded during the main loop (decode-sized tiles only):
  // row scales [32] and QKV routing [3][32]; the two-term BN = 16 variant
  // (O projection and down: residual epilogue) also residual rows [4][128]
  // and the next norm's gains [128]; the one-term BN = 32 variant (the QKV
  // projection with its context rows) the q/k-norm gains [128] and the RoPE
  // (cos, sin) of its rows [4][64].
  static constexpr bool PRE = BN <= 32;
  static constexpr bool PRE_RESID = PRE && SPLIT && BN == 16;
  static constexpr bool PRE_ROPE = PRE && !SPLIT && BN == 32;
  static constexpr int PRE_OFF = MAIN_BYTES + 256;
  static constexpr int PRE_BYTES = !PRE ? 0 : ((PRE_RESID || PRE_ROPE) ? 3072 : 512);
  static constexpr int PRE_RESID_ROWS = 4;
  // row scales 1/rms of the m-tile's rows (deferred input RMSNorm), computed
  // during the main loop and applied where each accumulator is last written
  static constexpr int RINV_OFF = MAIN_BYTES + 256 + PRE_BYTES;
  static constexpr int SMEM_BYTES = RINV_OFF + BN * 4 + 1024;  // + alignment slack
  static constexpr int TMEM_COLS = BN < 32 ? 32 : BN;
};

// 1/rms of rows m0 .. m0+rows-1 of the deferred input RMSNorm into out[]:
// the row's per-tile sums of squares in one fixed order for any M
// (accumulator i takes tiles i, i+32, ...; the 32 accumulators then combine
// halves, quarters, ... as an xor butterfly across a warp would), 1 for rows
// past norm_rows.  Thread t of nt takes rows t, t+nt, ...
__device__ void row_scales(const GemmParams& p, int m0, int rows, float* out, int t, int nt) {
  for (int r = t; r < rows; r += nt) {
    const float* q = p.ssq_in + static_cast<size_t>(m0 + r) * p.ssq_in_tiles;
    float acc[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) acc[i] = 0.f;
    for (int t0 = 0; t0 < p.ssq_in_tiles; t0 += 32) {
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (t0 + i < p.ssq_in_tiles) acc[i] += __ldcg(q + t0 + i);
    }
#pragma unroll
    for (int w = 16; w > 0; w >>= 1)
#pragma unroll
      for (int i = 0; i < w; ++i) acc[i] += acc[i + w];
    out[r] = (m0 + r < p.norm_rows) ? rsqrtf(acc[0] / static_cast<float>(p.norm_dim) + p.norm_eps) : 1.f;
  }
}

// ---------------------------------------------------------------- kernel
template <int BN, bool SPLIT>
__global__ void __launch_bounds__(128, 1)
    gemm_tc05_kernel(const __grid_constant__ CUtensorMap wmap,
                     const __grid_constant__ CUtensorMap xmap,
                     const __grid_constant__ CUtensorMap xmap_lo,
                     const __grid_constant__ GemmParams p) {
  using C = GemmCfg<BN, SPLIT>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::MAIN_BYTES);
  uint64_t* empty = full + C::STAGES;
  uint64_t* done = empty + C::STAGES;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* last_flag = reinterpret_cast<volatile int*>(tmem_slot + 2);
  float* ts = reinterpret_cast<float*>(smem);  // staged tile (after the mainloop)

  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  // grid (m-tiles, splits, n-tiles): the m-tiles of one weight tile are
  // consecutive CTAs (clusters), so they stream the same weight rows together
  // and the second one reads them from L2
  const int tile = blockIdx.z, split = blockIdx.y, mt = blockIdx.x;
  const int n_tiles = gridDim.z;
  const int m0 = mt * BN;
  const int kb0 = split * p.kb_per_split;
  const int kb1 = min(p.kb_total, kb0 + p.kb_per_split);
  const int nkb = kb1 - kb0;

  if (tid == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(done, 1);
    *abort_flag = 0;
    *last_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&wmap);
    tma_prefetch_desc(&xmap);
    if (SPLIT) tma_prefetch_desc(&xmap_lo);
  }
  if (warp == 1) tmem_alloc(tmem_slot, C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // The next kernel may launch once every CTA has signalled: at the start
  // (dep_lead < 0), or when this CTA's producer has dep_lead k-blocks left to
  // request, so that the next kernel's early weight loads follow this one's
  // instead of competing with them.
  if (p.dep_lead < 0 || nkb <= 0) griddep_launch_dependents();

  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer
    const uint64_t pol_w = l2_policy_evict_first();
    const uint64_t pol_x = l2_policy_evict_last();
    const int wrow = p.w_row0 + tile * p.w_tile_step;
    const int pre = nkb < C::STAGES ? nkb : C::STAGES;
    const int dep_it = p.dep_lead < 0 ? -1 : max(0, nkb - 1 - p.dep_lead);
    for (int it = 0; it < pre; ++it) {
      if (it == dep_it) griddep_launch_dependents();
      uint8_t* a = smem + it * C::A_BYTES;
      const int kx = (kb0 + it) * kTileK;
      mbar_arrive_expect_tx(&full[it], C::STAGE_BYTES);
      tma_load_2d(a, &wmap, kx, wrow, &full[it], pol_w);
      tma_load_2d(a + C::A_BYTES / 2, &wmap, kx, wrow + p.w_half_gap, &full[it], pol_w);
    }
    griddep_wait();  // activations come from the previous kernel
    for (int it = 0; it < pre; ++it) {
      uint8_t* b = smem + C::STAGES * C::A_BYTES + it * C::B_STAGE;
      tma_load_2d(b, &xmap, (kb0 + it) * kTileK, m0, &full[it], pol_x);
      if (SPLIT) tma_load_2d(b + C::B_BYTES, &xmap_lo, (kb0 + it) * kTileK, m0, &full[it], pol_x);
    }
    for (int it = pre; it < nkb; ++it) {
      const int s = it % C::STAGES;
      const uint32_t ph = ((it / C::STAGES) & 1) ^ 1;
      if (!mbar_wait(&empty[s], ph, abort_flag)) {
        *abort_flag = 1;
        raise_status(p.status, DFLASH_ERR_TIMEOUT, 11);
        griddep_launch_dependents();
        break;
      }
      if (it == dep_it) griddep_launch_dependents();
      uint8_t* a = smem + s * C::A_BYTES;
      uint8_t* b = smem + C::STAGES * C::A_BYTES + s * C::B_STAGE;
      const int kx = (kb0 + it) * kTileK;
      mbar_arrive_expect_tx(&full[s], C::STAGE_BYTES);
      tma_load_2d(a, &wmap, kx, wrow, &full[s], pol_w);
      tma_load_2d(a + C::A_BYTES / 2, &wmap, kx, wrow + p.w_half_gap, &full[s], pol_w);
      tma_load_2d(b, &xmap, kx, m0, &full[s], pol_x);
      if (SPLIT) tma_load_2d(b + C::B_BYTES, &xmap_lo, kx, m0, &full[s], pol_x);
    }
  } else if (warp == 1 && lane == 0) {
    // ---------------- MMA issuer (single thread)
    constexpr uint32_t idesc = umma_idesc_bf16(kTileN, BN);
    for (int it = 0; it < nkb; ++it) {
      const int s = it % C::STAGES;
      const uint32_t ph = (it / C::STAGES) & 1;
      if (!mbar_wait(&full[s], ph, abort_flag)) {
        *abort_flag = 1;
        raise_status(p.status, DFLASH_ERR_TIMEOUT, 12);
        break;
      }
      tc_fence_after();
      const uint64_t ad = umma_desc_sw128(smem_u32(smem + s * C::A_BYTES));
      const uint32_t b_addr = smem_u32(smem + C::STAGES * C::A_BYTES + s * C::B_STAGE);
      const uint64_t bd = umma_desc_sw128(b_addr);
#pragma unroll
      for (int k = 0; k < kTileK / 16; ++k) {
        umma_bf16(tmem, ad + 2 * k, bd + 2 * k, idesc, (it | k) != 0 ? 1u : 0u);
        // W x_lo into the same accumulator: W (x_hi + x_lo)
        if (SPLIT) umma_bf16(tmem, ad + 2 * k, umma_desc_sw128(b_addr + C::B_BYTES) + 2 * k, idesc, 1u);
      }
      umma_commit(&empty[s]);
    }
    umma_commit(done);
  }
  if (!(warp == 0 && lane == 0)) griddep_wait();
  __syncwarp();

  // ---------------- epilogue inputs, loaded by warps 2-3 (idle in the main
  // loop) once the previous kernels' writes are visible, so that the tail
  // after the last MMA starts with them in shared memory.  Same values and
  // the same arithmetic as the epilogue's own loads.
  float* rinv_s = reinterpret_cast<float*>(smem + C::RINV_OFF);          // [BN]
  int* pre_route = reinterpret_cast<int*>(smem + C::PRE_OFF + 128);      // [3][32]
  float* pre_resid = reinterpret_cast<float*>(smem + C::PRE_OFF + 512);  // [4][128]
  float* pre_g = pre_resid + C::PRE_RESID_ROWS * kTileN;                 // [128]
  float* pre_qg = reinterpret_cast<float*>(smem + C::PRE_OFF + 512);    // [128]
  float2* pre_cs = reinterpret_cast<float2*>(smem + C::PRE_OFF + 1024);  // [4][64]
  const int rows_mt = min(BN, p.M - mt * BN);                            // rows of this m-tile
  bool have_route = false, have_resid = false, have_rope = false;
  const bool rinv_early = p.ssq_in != nullptr && (p.pre_mask & 1);
  int rope_rb = 0;  // first row (in the m-tile) of the RoPE table
  if (rinv_early && warp >= 2) {
    if (BN <= 32) {
      // decode-sized tiles: lane t adds tiles t, t+32, ... of rows w2, w2+2,
      // ..., then the xor butterfly of warp_sum (the same sums as row_scales)
      const int w2 = warp - 2;
      float acc[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) acc[i] = 0.f;
      for (int tt = lane; tt < p.ssq_in_tiles; tt += 32) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int r = w2 + 2 * i;
          if (r < rows_mt) acc[i] += __ldcg(p.ssq_in + static_cast<size_t>(m0 + r) * p.ssq_in_tiles + tt);
        }
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int r = w2 + 2 * i;
        if (r < rows_mt) {
          const float ss = warp_sum(acc[i]);
          if (lane == 0)
            rinv_s[r] = (m0 + r < p.norm_rows) ? rsqrtf(ss / static_cast<float>(p.norm_dim) + p.norm_eps) : 1.f;
        }
      }
    } else {
      row_scales(p, m0, rows_mt, rinv_s, tid - 64, 64);
    }
  }
  if constexpr (C::PRE) {
    have_route = p.mode == EPI_QKV && (p.pre_mask & 2);
    if constexpr (C::PRE_ROPE) {
      // the rows this CTA will finish, as decided after the main loop
      int rb = 0, rc = rows_mt;
      if (p.splits > 1) {
        if (p.cluster) {
          const int rpc = (rows_mt + p.splits - 1) / p.splits;
          rb = min(rows_mt, static_cast<int>(cluster_ctarank()) * rpc);
          rc = min(rows_mt, rb + rpc) - rb;
        } else {
          rc = C::PRE_RESID_ROWS + 1;
        }
      }
      // one head per 128-feature tile (head_dim 128): a single gain vector
      have_rope = have_route && (p.pre_mask & 8) && rc <= C::PRE_RESID_ROWS && p.qkv.head_dim == kTileN;
      rope_rb = rb;
    }
    if constexpr (C::PRE_RESID) {
      // the rows this CTA will finish (as decided below): all of them, or
      // its share of a split-K cluster
      int rb = 0, rc = rows_mt;
      if (p.splits > 1) {
        if (p.cluster) {
          int rpc = (rows_mt + p.splits - 1) / p.splits;
          if (p.conv != nullptr && p.conv_width > 0) rpc = (rpc + p.block - 1) / p.block * p.block;
          rb = min(rows_mt, static_cast<int>(cluster_ctarank()) * rpc);
          rc = min(rows_mt, rb + rpc) - rb;
        } else {
          rc = C::PRE_RESID_ROWS + 1;  // the finishing CTA is known only at the end
        }
      }
      have_resid = p.mode == EPI_RESID && (p.pre_mask & 4) && rc <= C::PRE_RESID_ROWS;
      if (have_resid && warp >= 2) {
        const int t = tid - 64;
        const int n0 = tile * kTileN;
        for (int idx = t; idx < rc * (kTileN / 4); idx += 64) {
          const int r = idx / (kTileN / 4), c4 = idx % (kTileN / 4);
          *reinterpret_cast<float4*>(pre_resid + r * kTileN + c4 * 4) = __ldcg(
              reinterpret_cast<const float4*>(p.resid + static_cast<size_t>(mt * BN + rb + r) * p.ld_resid + n0) + c4);
        }
        if (p.gnext != nullptr)
          for (int f = t; f < kTileN; f += 64) pre_g[f] = bf2f(p.gnext[n0 + f]);
      }
    }
    if (warp >= 2) {
      const int w2 = warp - 2;
      const int mt0 = mt * BN;
      if (have_route) {
        const int t = tid - 64;
        if (t < rows_mt) qkv_route(p, mt0 + t, pre_route + t, pre_route + 32 + t, pre_route + 64 + t);
      }
      if (have_rope) {
        // q/k-norm gains of this tile's head(s), and (cos, sin) of every
        // rotate-half pair at the position of each row this CTA finishes
        // (the same rope_sincos the epilogue would call)
        const QkvEpi& e = p.qkv;
        const int t = tid - 64;
        const int d = e.head_dim, half = d / 2;
        const int head = (e.f0 + tile * kTileN) / d;
        const uint16_t* gsrc = head < e.n_q_heads ? e.q_norm
                               : (head < e.n_q_heads + e.n_kv_heads ? e.k_norm : nullptr);
        for (int f = t; f < d; f += 64) pre_qg[f] = gsrc != nullptr ? bf2f(gsrc[f]) : 1.f;
        asm volatile("bar.sync 1, 64;" ::: "memory");  // routing of all rows written (warps 2-3)
        int rc = min(C::PRE_RESID_ROWS, rows_mt - rope_rb);
        for (int idx = t; idx < rc * half; idx += 64) {
          const int r = idx / half, pr = idx % half;
          float sn, cs;
          rope_sincos(pre_route[32 + rope_rb + r], e.rope[pr], &sn, &cs);
          pre_cs[r * 64 + pr] = make_float2(cs, sn);
        }
      }
    }
  }

  // ---------------- epilogue: TMEM -> (partials | staged tile)
  const bool ok = mbar_wait(done, 0, abort_flag);
  if (!ok) {
    *abort_flag = 1;
    if (lane == 0) raise_status(p.status, DFLASH_ERR_TIMEOUT, 13);
  }
  __syncthreads();
  const bool aborted = *abort_flag != 0;
  tc_fence_after();
  const int rows = min(BN, p.M - m0);
  const bool scaled = p.ssq_in != nullptr;  // rows carry the input norm's 1/rms
  if (scaled && !rinv_early) {
    row_scales(p, m0, rows, rinv_s, tid, 128);
    __syncthreads();
  }
  const int f = warp * 32 + lane;
  const int n0 = tile * kTileN;
  bool do_epi = false;
  // rows of the tile this CTA finishes: all of them without split-K; with
  // split-K the S CTAs of the tile form one cluster and CTA q finishes rows
  // [q*rpc, q*rpc + rpc) (request-aligned when the block conv couples rows)
  int r_beg = 0, r_cnt = rows;
  bool push = false;  // split-K partials pushed to their owners (no final barrier)
  if (p.splits == 1) {
    if (!aborted) {
#pragma unroll 1
      for (int c = 0; c < BN / 16; ++c) {
        float v[16];
        tmem_ld16(tmem + (static_cast<uint32_t>(warp * 32) << 16) + c * 16, v);
        if (scaled) {
          // the chunk's 16 row scales, read before any of its stores
          float sc[16];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float4 t4 = *reinterpret_cast<const float4*>(rinv_s + c * 16 + 4 * q);
            sc[4 * q] = t4.x; sc[4 * q + 1] = t4.y; sc[4 * q + 2] = t4.z; sc[4 * q + 3] = t4.w;
          }
#pragma unroll
          for (int j = 0; j < 16; ++j) v[j] = (c * 16 + j < rows) ? v[j] * sc[j] : v[j];
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) ts[(c * 16 + j) * C::TS_LD + f] = v[j];
      }
      do_epi = true;
    }
    // thread f staged feature column f; the epilogues read across columns
    __syncthreads();
  } else if (!p.cluster) {
    // Split-K through global memory: every CTA stores its fp32 partial tile;
    // the last CTA of the tile (atomic ticket, no waiting) sums the partials
    // in split order and finishes the whole tile.
    if (!aborted) {
      float* part = p.partial + static_cast<size_t>(split) * p.M * p.N;
#pragma unroll 1
      for (int c = 0; c < BN / 16; ++c) {
        float v[16];
        tmem_ld16(tmem + (static_cast<uint32_t>(warp * 32) << 16) + c * 16, v);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int r = c * 16 + j;
          if (r < rows) part[static_cast<size_t>(m0 + r) * p.N + n0 + f] = v[j];
        }
      }
      __threadfence();
    }
    __syncthreads();
    if (tid == 0) {
      const int prev = aborted ? 0 : atomicAdd(&p.counters[mt * n_tiles + tile], 1);
      *last_flag = (!aborted && prev == p.splits - 1) ? 1 : 0;
    }
    __syncthreads();
    if (*last_flag) {
      __threadfence();
      const size_t sstride = static_cast<size_t>(p.M) * p.N / 4;  // float4 per split
      const float4* pbase = reinterpret_cast<const float4*>(p.partial);
      const int nchunk = rows * 32;
      for (int c0 = tid; c0 < nchunk; c0 += 4 * 128) {
        // up to 4 chunks per thread, splits in groups of 4: 16 loads in flight
        const float4* src[4];
        float4 acc[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int c = c0 + i * 128;
          src[i] = pbase + (static_cast<size_t>(m0 + (c < nchunk ? c / 32 : 0)) * p.N + n0) / 4 + c % 32;
          acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        int sp = 0;
        for (; sp + 4 <= p.splits; sp += 4) {
          float4 v[4][4];
#pragma unroll
          for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j)
              v[i][j] = (c0 + i * 128 < nchunk) ? __ldcg(src[i] + (sp + j) * sstride)
                                               : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
          for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              acc[i].x += v[i][j].x; acc[i].y += v[i][j].y;
              acc[i].z += v[i][j].z; acc[i].w += v[i][j].w;
            }
        }
        for (; sp < p.splits; ++sp) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            if (c0 + i * 128 < nchunk) {
              const float4 v = __ldcg(src[i] + sp * sstride);
              acc[i].x += v.x; acc[i].y += v.y; acc[i].z += v.z; acc[i].w += v.w;
            }
          }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int c = c0 + i * 128;
          if (c < nchunk) {
            if (scaled) {
              const float sc = rinv_s[c / 32];
              acc[i].x *= sc; acc[i].y *= sc; acc[i].z *= sc; acc[i].w *= sc;
            }
            *reinterpret_cast<float4*>(ts + (c / 32) * C::TS_LD + (c % 32) * 4) = acc[i];
          }
        }
      }
      if (tid == 0) p.counters[mt * n_tiles + tile] = 0;
      __syncthreads();
      do_epi = true;
    }
  } else {
    // 1) own partial tile -> own shared memory
    if (!aborted) {
#pragma unroll 1
      for (int c = 0; c < BN / 16; ++c) {
        float v[16];
        tmem_ld16(tmem + (static_cast<uint32_t>(warp * 32) << 16) + c * 16, v);
#pragma unroll
        for (int j = 0; j < 16; ++j) ts[(c * 16 + j) * C::TS_LD + f] = v[j];
      }
    }
    const int S = p.splits;
    const int q = static_cast<int>(cluster_ctarank());
    int rpc = (rows + S - 1) / S;
    if (p.conv != nullptr && p.conv_width > 0) rpc = (rpc + p.block - 1) / p.block * p.block;
    r_beg = min(rows, q * rpc);
    r_cnt = min(rows, r_beg + rpc) - r_beg;
    // Push when the partials of this CTA's rows fit its receive area (same
    // decision in every CTA of the cluster: same tile rows and splits)
    push = C::RECV_OFF + S * rpc * kTileN * 4 <= C::MAIN_BYTES;
    if (push) {
      __syncthreads();
      cluster_sync();  // every peer has drained its pipeline: receive areas are free
      // 2) each row of the tile -> slot [split] of the CTA that finishes it
      const uint32_t recv_addr = smem_u32(smem + C::RECV_OFF);
      for (int c = tid; c < rows * 32; c += 128) {
        const int r = c / 32, c4 = c % 32;
        const int own = r / rpc, lr = r % rpc;
        const float4 v = *reinterpret_cast<const float4*>(ts + r * C::TS_LD + c4 * 4);
        const uint32_t dst = dsmem_map(recv_addr + static_cast<uint32_t>(((split * rpc + lr) * 32 + c4) * 16),
                                       static_cast<uint32_t>(own));
        asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "f"(v.x), "f"(v.y),
                     "f"(v.z), "f"(v.w)
                     : "memory");
      }
      cluster_sync();  // all partials delivered
      // 3) sum this CTA's rows over the splits in split order (local reads)
      const float4* recv = reinterpret_cast<const float4*>(smem + C::RECV_OFF);
      for (int c = tid; c < r_cnt * 32; c += 128) {
        const int lr = c / 32, c4 = c % 32;
        float4 acc = recv[lr * 32 + c4];
        for (int sp = 1; sp < S; ++sp) {
          const float4 v = recv[(sp * rpc + lr) * 32 + c4];
          acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
        }
        if (scaled) {
          const float sc = rinv_s[r_beg + lr];
          acc.x *= sc; acc.y *= sc; acc.z *= sc; acc.w *= sc;
        }
        *reinterpret_cast<float4*>(ts + (r_beg + lr) * C::TS_LD + c4 * 4) = acc;
      }
      __syncthreads();
      do_epi = !aborted && r_cnt > 0;
    } else {
      cluster_sync();
      // 2) reduce this CTA's rows over the cluster's partials (split order)
      // Peers read only rows of their own range from this CTA's tile and this
      // CTA overwrites only rows of its range, so the in-place write needs no
      // extra barrier; the final cluster barrier keeps every tile alive until
      // all peers are done reading.
      const uint32_t ts_addr = smem_u32(ts);
      const int nchunk = r_cnt * 32;  // float4 chunks of my rows
      for (int c0 = tid; c0 < nchunk; c0 += 4 * 128) {
        float4 red[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) red[i] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
        for (int sp = 0; sp < S; ++sp) {
          const uint32_t peer = dsmem_map(ts_addr, static_cast<uint32_t>(sp));
          float4 v[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int c = c0 + i * 128;
            v[i] = c < nchunk
                       ? dsmem_ld4(peer + static_cast<uint32_t>(((r_beg + c / 32) * C::TS_LD + (c % 32) * 4) * 4))
                       : make_float4(0.f, 0.f, 0.f, 0.f);
          }
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            red[i].x += v[i].x; red[i].y += v[i].y; red[i].z += v[i].z; red[i].w += v[i].w;
          }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int c = c0 + i * 128;
          if (c < nchunk) {
            if (scaled) {
              const float sc = rinv_s[r_beg + c / 32];
              red[i].x *= sc; red[i].y *= sc; red[i].z *= sc; red[i].w *= sc;
            }
            *reinterpret_cast<float4*>(ts + (r_beg + c / 32) * C::TS_LD + (c % 32) * 4) = red[i];
          }
        }
      }
      __syncthreads();
      do_epi = !aborted && r_cnt > 0;
    }
  }
  float* tsv = ts + r_beg * C::TS_LD;   // first row this CTA finishes
  const int m0v = m0 + r_beg;
  const int rows_v = r_cnt;
  if (do_epi) {
    CtaSync sync;
    switch (p.mode) {
      case EPI_STORE_BF16:
      case EPI_STORE_F32: epi_store(p, tsv, tile, m0v, rows_v, tid, sync); break;
      case EPI_RESID:
        epi_resid(p, tsv, tile, m0v, rows_v, tid, sync, have_resid ? pre_resid : nullptr,
                  have_resid && p.gnext != nullptr ? pre_g : nullptr);
        break;
      case EPI_SWIGLU: epi_swiglu(p, tsv, tile, m0v, rows_v, tid, sync); break;
      case EPI_ARGMAX: epi_argmax(p, tsv, tile, m0v, rows_v, tid, sync, n_tiles); break;
      case EPI_QKV:
        epi_qkv(p, tsv, tile, m0v, rows_v, reinterpret_cast<int*>(smem + C::SCRATCH_OFF + BN * 4), BN,
                tid, sync, have_route ? pre_route + r_beg : nullptr, 32,
                have_rope && r_beg == rope_rb ? pre_qg : nullptr,
                have_rope && r_beg == rope_rb ? pre_cs : nullptr);
        break;
      default: break;
    }
  }
  if (p.mode == EPI_ARGMAX && p.amax_key != nullptr) {
    // the last CTA to finish turns the per-row keys into tokens (no waiting:
    // every other CTA has folded its keys in before taking its ticket)
    __threadfence();
    __syncthreads();
    if (tid == 0) {
      const int n_ctas = gridDim.x * gridDim.y * gridDim.z;
      *last_flag = (atomicAdd(p.amax_ticket, 1) == n_ctas - 1) ? 1 : 0;
    }
    __syncthreads();
    if (*last_flag) {
      __threadfence();
      for (int r = tid; r < p.M; r += 128) {
        const int idx = argmax_key_index(atomicExch(p.amax_key + r, 0ull));
        const int i = r % p.amax_block;
        if (!p.amax_skip_first)
          p.amax_out[r] = idx;
        else if (i != 0)
          p.amax_out[(r / p.amax_block) * (p.amax_block - 1) + i - 1] = idx;
      }
      if (tid == 0) *p.amax_ticket = 0;
    }
  }
  if (p.splits > 1 && p.cluster && !push) cluster_sync();  // peers may still read this CTA's tile until here
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, C::TMEM_COLS);
}

// ---------------------------------------------------------------- host side
int gemm_bn_for(int M, int N, int sms) {
  if (M <= 128) return M <= 16 ? 16 : M <= 32 ? 32 : M <= 64 ? 64 : 128;
  // more rows: 256-row tiles, or 128-row tiles where 256-row tiles would
  // leave SMs without a tile (fewer output tiles than SMs)
  return (N / kTileN) * ((M + 255) / 256) < sms ? 128 : 256;
}

template <bool SPLIT>
static int max_smem_split() {
  int m = GemmCfg<16, SPLIT>::SMEM_BYTES;
  m = m > GemmCfg<32, SPLIT>::SMEM_BYTES ? m : GemmCfg<32, SPLIT>::SMEM_BYTES;
  m = m > GemmCfg<64, SPLIT>::SMEM_BYTES ? m : GemmCfg<64, SPLIT>::SMEM_BYTES;
  m = m > GemmCfg<128, SPLIT>::SMEM_BYTES ? m : GemmCfg<128, SPLIT>::SMEM_BYTES;
  m = m > GemmCfg<256, SPLIT>::SMEM_BYTES ? m : GemmCfg<256, SPLIT>::SMEM_BYTES;
  return m;
}
int gemm_max_smem_bytes() {
  const int a = max_smem_split<false>(), b = max_smem_split<true>();
  return a > b ? a : b;
}

// Dynamic shared memory size, and the largest shared-memory carveout so that
// several CTAs (of this and of the next kernel) can be resident per SM.
template <int BN, bool SPLIT>
static cudaError_t set_gemm_attrs() {
  cudaError_t e = cudaFuncSetAttribute(gemm_tc05_kernel<BN, SPLIT>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       GemmCfg<BN, SPLIT>::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(gemm_tc05_kernel<BN, SPLIT>,
                           cudaFuncAttributePreferredSharedMemoryCarveout,
                           cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  // split-K clusters of up to 16 CTAs (non-portable size, supported on sm_103)
  return cudaFuncSetAttribute(gemm_tc05_kernel<BN, SPLIT>,
                              cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
}

template <int BN, bool SPLIT>
static cudaError_t launch_bn(const CUtensorMap* w_map, const CUtensorMap* x_map,
                             const CUtensorMap* x_lo_map, const GemmParams& p, cudaStream_t s,
                             bool pdl) {
  using C = GemmCfg<BN, SPLIT>;
  static thread_local int attr_device = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (attr_device != dev) {
    cudaError_t e = set_gemm_attrs<BN, SPLIT>();
    if (e != cudaSuccess) return e;
    attr_device = dev;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((p.M + BN - 1) / BN, p.splits, p.N / kTileN);
  cfg.blockDim = dim3(128, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = s;
  cudaLaunchAttribute attr[3];
  int na = 0;
  if (pdl) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  if (p.splits > 1 && p.cluster) {
    // the split-K CTAs of one output tile form a cluster (reduced through DSMEM)
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = 1;
    attr[na].val.clusterDim.y = p.splits;
    attr[na].val.clusterDim.z = 1;
    ++na;
    // let several CTAs of a cluster share an SM, so clusters of 8 do not cap
    // the number of resident CTAs
    attr[na].id = cudaLaunchAttributeClusterSchedulingPolicyPreference;
    attr[na].val.clusterSchedulingPolicyPreference = cudaClusterSchedulingPolicyLoadBalancing;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  count_launch();
  return cudaLaunchKernelEx(&cfg, gemm_tc05_kernel<BN, SPLIT>, *w_map, *x_map, *x_lo_map, p);
}

template <int BN>
static int max_clusters_bn(int cluster) {
  using C = GemmCfg<BN, false>;
  if (set_gemm_attrs<BN, false>() != cudaSuccess) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1, cluster, 1);
  cfg.blockDim = dim3(128, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = cluster;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, gemm_tc05_kernel<BN, false>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

int gemm_max_active_clusters(int bn, int cluster) {
  switch (bn) {
    case 16: return max_clusters_bn<16>(cluster);
    case 32: return max_clusters_bn<32>(cluster);
    case 64: return max_clusters_bn<64>(cluster);
    case 128: return max_clusters_bn<128>(cluster);
    case 256: return max_clusters_bn<256>(cluster);
    default: return 0;
  }
}

cudaError_t gemm_launch(const CUtensorMap* w_map, const CUtensorMap* x_map,
                        const CUtensorMap* x_lo_map, const GemmParams& p, int bn, cudaStream_t s,
                        bool pdl) {
  if (x_lo_map != nullptr) {
    switch (bn) {
      case 16: return launch_bn<16, true>(w_map, x_map, x_lo_map, p, s, pdl);
      case 32: return launch_bn<32, true>(w_map, x_map, x_lo_map, p, s, pdl);
      case 64: return launch_bn<64, true>(w_map, x_map, x_lo_map, p, s, pdl);
      case 128: return launch_bn<128, true>(w_map, x_map, x_lo_map, p, s, pdl);
      case 256: return launch_bn<256, true>(w_map, x_map, x_lo_map, p, s, pdl);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (bn) {
    case 16: return launch_bn<16, false>(w_map, x_map, x_map, p, s, pdl);
    case 32: return launch_bn<32, false>(w_map, x_map, x_map, p, s, pdl);
    case 64: return launch_bn<64, false>(w_map, x_map, x_map, p, s, pdl);
    case 128: return launch_bn<128, false>(w_map, x_map, x_map, p, s, pdl);
    case 256: return launch_bn<256, false>(w_map, x_map, x_map, p, s, pdl);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace dflash
