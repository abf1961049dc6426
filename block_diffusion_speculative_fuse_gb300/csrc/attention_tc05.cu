// Drafter attention on the 5th-generation tensor cores (tcgen05, sm_103a).
//
// The block rows of a request attend, without a mask, to every context key
// of the paged pool and to every key of the block itself (DFlash-2
// mechanisms: the drafter is non-causal).  One CTA = (request, KV head, key
// split); the key splits of a (request, KV head) form one thread-block
// cluster (<= 16 CTAs) and merge their partial (O, m, l) through distributed
// shared memory.
//
// Query rows: the G = hq/hkv query heads that share the KV head times the n
// block rows, row index i*G + h (R = n*G rows).  Keys are streamed in chunks
// of 64 (four 16-key pages) by TMA into a 4-deep ring of 128-byte-swizzled
// stages.  A K plane is laid out [64-column half][64 keys][128 B] (the S MMA
// reads all 64 keys of a column slice at once), filled by one box per (page,
// half); a V plane [page][half][16 keys][128 B] (the PV MMA reads one page
// per instruction), filled by one box per page.  The SM's TMA unit spends a
// roughly fixed time per box, so fewer, larger boxes keep it ahead of HBM.
// Pages past the split or missing from the table are read from beyond the
// end of the tensor map, which fills them with zeros.
//
// Per chunk c (warp 5 lane 0 issues, fp32 accumulators in TMEM):
//   S[c%2] = Q K^T            M = 128 rows, N = 64 keys, K = head_dim
//   O     += P[c%2] V         M = 128 rows, N = head_dim, K = 64 keys
// Warps 0-3 own TMEM lanes 32w..32w+31.  Each thread reads its S row, masks
// invalid keys and forms P = exp2(t - m) in the exp2 domain with a lazily
// updated row maximum m: O and l are rescaled only when a chunk's maximum
// exceeds m by more than 2^8 (so P <= 256), which keeps O in TMEM across
// chunks.  P is stored in shared memory as the K-major A operand of the PV
// MMA; V is the MN-major B operand.
//
// Two warp pairs (R <= 64): the query tile holds the R rows twice (MMA rows
// 0-63 and 64-127), so every S tile carries the scores in both TMEM halves.
// Warps 0-1 take the even chunks (lanes 0-63), warps 2-3 the odd chunks
// (lanes 64-127); P[0] keeps rows 64-127 zero and P[1] rows 0-63, so the
// even chunks accumulate into O lanes 0-63 and the odd ones into lanes
// 64-127, two independent online-softmax states that are merged like key
// splits.  With R > 64 all four warps take every chunk (one state).
#include "common.cuh"
#include "kernels.h"

namespace dflash {

namespace {

constexpr int kChunkKeys = 64;
constexpr int kChunkPages = 4;
constexpr int kMaxPagesTc = 1024;  // pages per split (staged ids)
// causal (target) key splits: fixed 512-key boundaries, so a row's result
// does not depend on the batch or the number of rows of the call
constexpr int kTargetSplitPagesTc = 32;
constexpr float kRescaleLog2 = 8.f;
constexpr int kThreads = 192;      // warps 0-3 softmax, 4 TMA, 5 MMA

// TERMS = 2: every key chunk also carries the low bf16 terms of K and V
// (planes K, V, K_lo, V_lo in a stage, as in the pool's pages).
// FP8: the context pages hold E4M3 codes and per-vector scales; they arrive
// in a ring of code stages and eight converter warps turn them into the bf16
// stages the MMAs read (block keys arrive there as bf16 directly).
template <int D, int TERMS = 1, bool FP8 = false>
struct TcCfg {
  static constexpr int CONV_THREADS = 256;        // FP8: warps 6-13 convert
  static constexpr int THREADS = FP8 ? 192 + CONV_THREADS : 192;
  static constexpr int STAGES = TERMS == 2 ? 2 : (FP8 ? 3 : 4);
  static constexpr int F8_STAGES = FP8 ? 3 : 0;
  static constexpr int K8_BYTES = kChunkKeys * D;               // [64 keys][D] codes
  static constexpr int F8_STAGE_BYTES = 2 * K8_BYTES;           // K codes then V codes
  static constexpr int SC_BYTES = 2 * kChunkKeys * 4;           // K scales then V scales
  static constexpr int PLANES = 2 * TERMS;
  static constexpr int HALVES = D / 64;
  static constexpr int Q_BYTES = 128 * D * 2;                   // [HALVES][128 rows][64]
  static constexpr int P_BYTES = 128 * kChunkKeys * 2;          // [128 rows][64 keys]
  static constexpr int KV_HALF = kChunkKeys * 64 * 2;           // K plane: [64 keys][64 cols] = 8 KB
  static constexpr int K_BYTES = kChunkKeys * D * 2;            // one plane (K: [HALVES][64][64])
  static constexpr int PH_BYTES = 16 * 128;                     // V plane: 16 keys of one half
  static constexpr int PPL_BYTES = HALVES * PH_BYTES;           // V plane: one page [HALVES][16][64]
  static constexpr int STAGE_BYTES = PLANES * K_BYTES;          // K, V (, K_lo, V_lo)
  static constexpr int K_BOXES = kChunkPages * TERMS * HALVES;  // TMA boxes per chunk: K planes
  static constexpr int BOXES = K_BOXES + kChunkPages * TERMS;   // + one per page and V plane
  static constexpr int Q_OFF = 0;
  static constexpr int P_OFF = Q_OFF + Q_BYTES;
  static constexpr int KV_OFF = P_OFF + 2 * P_BYTES;
  static constexpr int F8_OFF = KV_OFF + STAGES * STAGE_BYTES;       // code ring
  static constexpr int SC8_OFF = F8_OFF + F8_STAGES * F8_STAGE_BYTES;  // scales of the code ring
  static constexpr int SCB_OFF = SC8_OFF + F8_STAGES * SC_BYTES;      // scales of the bf16 stages
  static constexpr int PG_OFF = SCB_OFF + (FP8 ? STAGES * SC_BYTES : 0);
  static constexpr int PN_OFF = PG_OFF + kMaxPagesTc * 4;
  static constexpr int BAR_OFF = PN_OFF + kMaxPagesTc * 4;
  static constexpr int SMEM = BAR_OFF + 512 + 1024;             // barriers + alignment slack
  // combine staging (after the key loop, in the K/V stage area): 128 row slots
  // merge staging: at most 160 partial rows (rows per CTA x parts x splits
  // <= (R + splits) x parts) of D + 4 floats plus (m, l)
  static_assert(160 * ((D + 4) * 4 + 8) <= STAGES * STAGE_BYTES + F8_STAGES * F8_STAGE_BYTES,
                "merge staging must fit");
  static_assert(BOXES <= 32, "one TMA box per producer lane");
  static constexpr uint32_t TMEM_COLS = 256;                    // S0 | S1 | O
  static constexpr uint32_t S_COL0 = 0, O_COL = 128;
};

// v[i] for a run-time i in [0, 4) without indexing a local array
__device__ __forceinline__ int pick4(const int (&v)[4], int i) {
  return i == 0 ? v[0] : i == 1 ? v[1] : i == 2 ? v[2] : v[3];
}
__device__ __forceinline__ uint32_t swz128(int row, int chunk16) {
  return static_cast<uint32_t>(row * 128 + ((chunk16 ^ (row & 7)) << 4));
}
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// CAUSAL (the target's verify / decode pass): block row i of the CTA's query
// tile sits at position pos0 + i and attends to pool keys [0, pos0 + i] (its
// own K/V were written to the pool by the QKV epilogue); there are no
// separate block keys.  The CTA takes block rows [qt*rpt, (qt+1)*rpt) of its
// request (p.rows_per_tile), so a row's arithmetic never depends on how many
// rows the call has.
template <int D, bool CAUSAL = false, int TERMS = 1, bool FP8 = false>
__global__ void __launch_bounds__(TcCfg<D, TERMS, FP8>::THREADS, 1)
    attn_tc05_kernel(const __grid_constant__ CUtensorMap pool_map,
                     const __grid_constant__ CUtensorMap pool_v_map,
                     const __grid_constant__ CUtensorMap kblk_map,
                     const __grid_constant__ CUtensorMap vblk_map,
                     const __grid_constant__ AttnTcParams p) {
  using C = TcCfg<D, TERMS, FP8>;
  static_assert(!FP8 || (!CAUSAL && TERMS == 1), "E4M3 context caches: drafter, one term");
  constexpr int kStages = C::STAGES;
  constexpr int kThreads = C::THREADS;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  uint64_t* kv_full = reinterpret_cast<uint64_t*>(sm + C::BAR_OFF);
  uint64_t* kv_empty = kv_full + kStages;
  uint64_t* s_full = kv_empty + kStages;  // [2]
  uint64_t* s_free = s_full + 2;          // [2]
  uint64_t* p_full = s_free + 2;          // [2]
  uint64_t* pv_done = p_full + 2;         // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(pv_done + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  uint64_t* f8_full = reinterpret_cast<uint64_t*>(sm + C::BAR_OFF + 256);  // FP8: code ring
  uint64_t* f8_empty = f8_full + 4;
  int* pages_s = reinterpret_cast<int*>(sm + C::PG_OFF);   // pool page, -1 none, <= -2 block page
  int* pages_n = reinterpret_cast<int*>(sm + C::PN_OFF);   // valid keys of each staged page

  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int split = blockIdx.x;
  const int req = blockIdx.y / p.hkv, g = blockIdx.y % p.hkv;
  const int G = p.hq / p.hkv;
  const int i0 = blockIdx.z * p.rows_per_tile;  // first block row of this query tile
  const int n_here = max(0, min(p.n, i0 + p.rows_per_tile) - i0);
  const int R = n_here * G;                     // real query rows (<= 128)
  const bool dual = R <= 64;                    // two warp pairs, two softmax states
  const int n_act = (R + 31) / 32;              // warps (per pair when dual) with real rows

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      // FP8: a bf16 stage is complete when every converter warp has arrived
      // (and the bf16 block keys they requested have landed)
      mbar_init(&kv_full[s], FP8 ? C::CONV_THREADS / 32 : 1);
      mbar_init(&kv_empty[s], 1);
    }
    for (int s = 0; s < C::F8_STAGES; ++s) {
      mbar_init(&f8_full[s], 1);
      mbar_init(&f8_empty[s], C::CONV_THREADS / 32);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&s_full[b], 1);
      mbar_init(&s_free[b], n_act);
      mbar_init(&p_full[b], n_act);
      mbar_init(&pv_done[b], 1);
    }
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&pool_map);
    if (!FP8) tma_prefetch_desc(&pool_v_map);
    tma_prefetch_desc(&kblk_map);
    tma_prefetch_desc(&vblk_map);
  }
  if (warp == 5) tmem_alloc(tmem_slot, C::TMEM_COLS);
  // both P buffers start at zero: rows that no thread writes stay zero
  for (int idx = tid; idx < 2 * C::P_BYTES / 16; idx += kThreads)
    *reinterpret_cast<uint4*>(sm + C::P_OFF + idx * 16) = make_uint4(0u, 0u, 0u, 0u);
  // The next kernel may launch once every CTA has issued its key loads (the
  // producer signals below), so that its early weight loads queue behind them.
  griddep_wait();

  // ---- one round of global loads, all issued before any is used: the
  //      context length, this split's page ids (read before the length is
  //      known) and the query rows
  constexpr int QCH = D / 8;                                  // 16-byte pieces per row
  constexpr int QMAX = (128 * QCH + kThreads - 1) / kThreads;
  constexpr int PMAX = (kMaxPagesTc + kThreads - 1) / kThreads;
  const int pg_lo = split * p.split_pages;
  const int L = __ldcg(p.pos0 + req);
  int pid[PMAX];
#pragma unroll
  for (int k = 0; k < PMAX; ++k) {
    const int i = tid + k * kThreads, j = pg_lo + i;
    pid[k] = (i < p.split_pages && j < p.max_pages)
                 ? __ldcg(p.page_table + static_cast<size_t>(req) * p.max_pages + j)
                 : -1;
  }
  const int qrows = dual ? 64 : 128;  // distinct tile rows (dual: rows 64-127 repeat 0-63)
  uint4 qv[QMAX];
#pragma unroll
  for (int k = 0; k < QMAX; ++k) {
    const int idx = tid + k * kThreads;
    const int row = idx / QCH, c = idx % QCH;
    qv[k] = make_uint4(0u, 0u, 0u, 0u);
    if (idx < qrows * QCH && row < R) {
      const int i = i0 + row / G, h = row % G;
      qv[k] = __ldcg(reinterpret_cast<const uint4*>(
          p.q + ((static_cast<size_t>(req) * p.n + i) * p.hq + g * G + h) * D + c * 8));
    }
  }
#pragma unroll
  for (int k = 0; k < QMAX; ++k) {
    const int idx = tid + k * kThreads;
    const int row = idx / QCH, c = idx % QCH;
    if (idx < qrows * QCH) {
      uint8_t* qb = sm + C::Q_OFF + (c / 8) * (128 * 128);
      *reinterpret_cast<uint4*>(qb + swz128(row, c % 8)) = qv[k];
      if (dual) *reinterpret_cast<uint4*>(qb + swz128(row + 64, c % 8)) = qv[k];
    }
  }
  // ---- key space of this request: context pages [0, Pc), then block pages
  // (causal: pool pages up to the tile's last row, no block pages)
  const int Lk = CAUSAL ? L + i0 + n_here : L;
  const int Pc = (Lk + 15) / 16;
  const int Pb = CAUSAL ? 0 : (p.n + 15) / 16;
  const int pg_hi = min(Pc + Pb, pg_lo + p.split_pages);
  const int npg = max(0, pg_hi - pg_lo);
  const int nch = (npg + kChunkPages - 1) / kChunkPages;
#pragma unroll
  for (int k = 0; k < PMAX; ++k) {
    const int i = tid + k * kThreads, j = pg_lo + i;
    if (i >= nch * kChunkPages) continue;
    int id = -1, cnt = 0;
    if (i < npg) {
      if (j < Pc) {
        id = pid[k];
        if (j >= p.max_pages || id < 0 || id >= p.n_pages) {
          raise_status(p.status, DFLASH_ERR_CAPACITY, 301);
          id = -1;
        } else {
          cnt = min(16, Lk - j * 16);
        }
      } else {
        id = -2 - (j - Pc);
        cnt = min(16, p.n - (j - Pc) * 16);
      }
    }
    pages_s[i] = id;
    pages_n[i] = cnt;
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (FP8 && warp == 4) {
    // ------------------------------------------------ E4M3 producer: codes (TMA) and
    // scales (bulk copies) of the context pages into the code ring
    const uint64_t pol = l2_policy_evict_first();
    constexpr int S8 = C::F8_STAGES > 0 ? C::F8_STAGES : 1;
    int issued = 0;
    for (int c = 0; c < nch; ++c) {
      const int st = c % S8;
      int n8 = 0;
#pragma unroll
      for (int pp = 0; pp < kChunkPages; ++pp) n8 += pages_s[c * kChunkPages + pp] >= 0 ? 1 : 0;
      int ok = 1;
      if (lane == 0) {
        if (c >= S8 && !mbar_wait(&f8_empty[st], ((c / S8) & 1) ^ 1, abort_flag)) {
          *abort_flag = 1;
          raise_status(p.status, DFLASH_ERR_TIMEOUT, 315);
          ok = 0;
        } else {
          mbar_arrive_expect_tx(&f8_full[st], n8 * 2 * (16 * D + 64));
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      if (lane < kChunkPages * 4) {
        // lane -> (page, K|V, codes|scales)
        const int pp = lane / 4, kv = (lane / 2) % 2, what = lane % 2;
        const int id = pages_s[c * kChunkPages + pp];
        if (id >= 0) {
          const int row = p.pool_row0 + ((id * 2 + kv) * p.hkv + g) * 16;  // first vector of the page
          if (what == 0)
            tma_load_2d(sm + C::F8_OFF + st * C::F8_STAGE_BYTES + kv * C::K8_BYTES + pp * 16 * D,
                        &pool_map, 0, row, &f8_full[st], pol);
          else
            bulk_load(sm + C::SC8_OFF + st * C::SC_BYTES + kv * (kChunkKeys * 4) + pp * 64,
                      p.scales + row, 64, &f8_full[st]);
        }
      }
      ++issued;
      if (c == min(nch, S8) - 1) griddep_launch_dependents();
    }
    if (nch == 0 || issued < min(nch, S8)) griddep_launch_dependents();  // none issued, or an abort
    if (lane == 0)
      for (int c = max(0, issued - S8); c < issued; ++c)
        mbar_wait(&f8_full[c % S8], (c / S8) & 1, nullptr);
  } else if (FP8 && warp >= 6) {
    // ------------------------------------------------ converters (warps 6..): code
    // stage -> bf16 stage (exact values; invalid keys as zeros), per-key
    // scales, and the bf16 block keys by TMA (first thread).  Thread t owns
    // the 8-code piece c8 = t % CH of key rows r0 + RPP*i (i = 0, 1, ...) of
    // K and of V, so a piece's page, its row within the page and its
    // 128-byte swizzle phase are fixed per thread; the page ids and valid
    // counts of the chunk are read once into registers.
    constexpr int S8 = C::F8_STAGES > 0 ? C::F8_STAGES : 1;
    constexpr int NT = C::CONV_THREADS;
    constexpr int CH = D / 8;                     // 8-code pieces per key row
    constexpr int RPP = NT / CH;                  // key rows per pass
    constexpr int JPK = kChunkKeys / RPP;         // passes per plane (K or V)
    static_assert(RPP % 8 == 0 && NT >= 2 * kChunkKeys, "converter thread mapping");
    const uint64_t pol = l2_policy_evict_first();
    const int t = tid - 192;
    const int c8 = t % CH, r0 = t / CH;
    const uint32_t f8_base = smem_u32(sm + C::F8_OFF) + r0 * D + c8 * 8;
    // row phase r0 % 8 = key % 8 for every key this thread writes (RPP % 8 == 0)
    const uint32_t k16_base = smem_u32(sm + C::KV_OFF) + r0 * 128 + (c8 / 8) * C::KV_HALF +
                              (((c8 % 8) ^ (r0 % 8)) << 4);
    const uint32_t v16_base = smem_u32(sm + C::KV_OFF + C::K_BYTES) + (c8 / 8) * C::PH_BYTES +
                              (((c8 % 8) ^ (r0 % 8)) << 4);
    int done_c = 0;
    for (int c = 0; c < nch; ++c) {
      const int st8 = c % S8, sb = c % kStages;
      bool ok = __all_sync(0xffffffffu, mbar_wait(&f8_full[st8], (c / S8) & 1, abort_flag));
      if (ok && c >= kStages)
        ok = __all_sync(0xffffffffu, mbar_wait(&kv_empty[sb], ((c / kStages) & 1) ^ 1, abort_flag));
      if (!ok) {
        *abort_flag = 1;
        if (lane == 0) raise_status(p.status, DFLASH_ERR_TIMEOUT, 316);
        break;
      }
      const int4 ids4 = *reinterpret_cast<const int4*>(pages_s + c * kChunkPages);
      const int4 cnt4 = *reinterpret_cast<const int4*>(pages_n + c * kChunkPages);
      const int idv[4] = {ids4.x, ids4.y, ids4.z, ids4.w};
      const int cnv[4] = {cnt4.x, cnt4.y, cnt4.z, cnt4.w};
      if (t == 0) {
        const int nb = (idv[0] <= -2) + (idv[1] <= -2) + (idv[2] <= -2) + (idv[3] <= -2);
        if (nb > 0) {
          mbar_expect_tx(&kv_full[sb], nb * 2 * C::HALVES * (16 * 64 * 2));
#pragma unroll
          for (int pp = 0; pp < kChunkPages; ++pp) {
            if (idv[pp] > -2) continue;
            const int y = (req * p.hkv + g) * p.n + (-2 - idv[pp]) * 16;
            uint8_t* kd = sm + C::KV_OFF + sb * C::STAGE_BYTES + pp * 16 * 128;
            for (int hf = 0; hf < C::HALVES; ++hf)
              tma_load_2d(kd + hf * C::KV_HALF, &kblk_map, hf * 64, y, &kv_full[sb], pol);
            tma_load_3d(sm + C::KV_OFF + sb * C::STAGE_BYTES + C::K_BYTES + pp * C::PPL_BYTES,
                        &vblk_map, 0, y, 0, &kv_full[sb], pol);
          }
        }
      }
      const uint32_t src = f8_base + st8 * C::F8_STAGE_BYTES;
      const uint32_t kdst = k16_base + sb * C::STAGE_BYTES;
      const uint32_t vdst = v16_base + sb * C::STAGE_BYTES;
#pragma unroll
      for (int j0 = 0; j0 < 2 * JPK; j0 += 8) {
        uint2 cd[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int j = j0 + u, kv = j / JPK, i = j % JPK;
          if (j >= 2 * JPK) break;
          cd[u] = ld_shared_u2(src + kv * C::K8_BYTES + RPP * i * D);
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int j = j0 + u, kv = j / JPK, i = j % JPK;
          if (j >= 2 * JPK) break;
          const int key = r0 + RPP * i, pp = key / 16;
          // RPP <= 16: the page is fixed by i; else r0 picks one of two pages
          const int id = RPP <= 16 ? idv[(RPP * i) / 16] : pick4(idv, pp);
          const int cnt = RPP <= 16 ? cnv[(RPP * i) / 16] : pick4(cnv, pp);
          if (id <= -2) continue;                      // block keys arrive as bf16
          uint4 o = make_uint4(0u, 0u, 0u, 0u);
          if (id >= 0 && key % 16 < cnt) {
            o = make_uint4(e4m3x2_to_bf16x2(cd[u].x), e4m3x2_to_bf16x2(cd[u].x >> 16),
                           e4m3x2_to_bf16x2(cd[u].y), e4m3x2_to_bf16x2(cd[u].y >> 16));
          }
          st_shared_u4(kv ? vdst + pp * C::PPL_BYTES + (key % 16) * 128 : kdst + RPP * i * 128, o);
        }
      }
      if (t < 2 * kChunkKeys) {
        // per-key scales of the stage (K then V): 0 past a page's valid keys,
        // 1 for block keys
        const int key = t % kChunkKeys, pp = key / 16;
        const int id = pick4(idv, pp), cnt = pick4(cnv, pp);
        const float* sc8 = reinterpret_cast<const float*>(sm + C::SC8_OFF + st8 * C::SC_BYTES);
        float v = 0.f;
        if (id <= -2)
          v = 1.f;
        else if (id >= 0 && key % 16 < cnt)
          v = sc8[t];
        reinterpret_cast<float*>(sm + C::SCB_OFF + sb * C::SC_BYTES)[t] = v;
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&f8_empty[st8]);
        mbar_arrive(&kv_full[sb]);
      }
      done_c = c + 1;
    }
    // block-key copies still in flight after an abort land before the CTA exits
    if (t == 0)
      for (int c = max(0, done_c - kStages); c < done_c; ++c)
        mbar_wait(&kv_full[c % kStages], (c / kStages) & 1, nullptr);
  } else if (warp == 4) {
    // ------------------------------------------------ TMA producer (one box per lane)
    const uint64_t pol = l2_policy_evict_first();
    int issued = 0;
    for (int c = 0; c < nch; ++c) {
      const int st = c % kStages;
      int ok = 1;
      if (lane == 0) {
        if (c >= kStages && !mbar_wait(&kv_empty[st], ((c / kStages) & 1) ^ 1, abort_flag)) {
          *abort_flag = 1;
          raise_status(p.status, DFLASH_ERR_TIMEOUT, 311);
          ok = 0;
        } else {
          mbar_arrive_expect_tx(&kv_full[st], C::STAGE_BYTES);
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      if (lane < C::BOXES) {
        // lanes [0, K_BOXES): (page, K term, 64-column half), one 2-D box each;
        // then (page, V term): both halves of the page's V rows in one 3-D box.
        // Planes of a pool page: K, V (, K_lo, V_lo).
        const bool kb = lane < C::K_BOXES;
        const int j = kb ? lane : lane - C::K_BOXES;
        const int pp = kb ? j / (TERMS * C::HALVES) : j / TERMS;
        const int t = kb ? (j / C::HALVES) % TERMS : j % TERMS;
        const int hf = kb ? j % C::HALVES : 0;
        const int kv = 2 * t + (kb ? 0 : 1);
        const int id = pages_s[c * kChunkPages + pp];
        bool blk = false;
        int y;
        if (id >= 0) {
          y = p.pool_row0 + ((id * C::PLANES + kv) * p.hkv + g) * 16;
        } else if (id <= -2) {
          blk = true;
          y = (req * p.hkv + g) * p.n + (-2 - id) * 16;
        } else {
          y = p.pool_rows;  // past the end: zero fill
        }
        uint8_t* dst = sm + C::KV_OFF + st * C::STAGE_BYTES + kv * C::K_BYTES;
        if (kb)
          tma_load_2d(dst + hf * C::KV_HALF + pp * 16 * 128, blk ? &kblk_map : &pool_map, hf * 64, y,
                      &kv_full[st], pol);
        else
          tma_load_3d(dst + pp * C::PPL_BYTES, blk ? &vblk_map : &pool_v_map, 0, y, 0, &kv_full[st],
                      pol);
      }
      ++issued;
      if (c == min(nch, kStages) - 1) griddep_launch_dependents();
    }
    if (nch == 0 || issued < min(nch, kStages)) griddep_launch_dependents();  // none issued, or an abort
    // copies still in flight after an abort land before the CTA exits
    if (lane == 0)
      for (int c = max(0, issued - kStages); c < issued; ++c)
        mbar_wait(&kv_full[c % kStages], (c / kStages) & 1, nullptr);
  } else if (warp == 5) {
    // ------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = umma_idesc_bf16(128, kChunkKeys);
      constexpr uint32_t idesc_pv = umma_idesc_bf16(128, D) | (1u << 16);  // B (V) MN-major
      const uint32_t q_addr = smem_u32(sm + C::Q_OFF);
      auto issue_s = [&](int c) -> bool {
        const int st = c % kStages, b = c & 1;
        if (!mbar_wait(&kv_full[st], (c / kStages) & 1, abort_flag)) return false;
        if (c >= 2 && !mbar_wait(&s_free[b], ((c - 2) >> 1) & 1, abort_flag)) return false;
        tc_fence_after();
        const uint32_t k_addr = smem_u32(sm + C::KV_OFF + st * C::STAGE_BYTES);
#pragma unroll
        for (int t = 0; t < TERMS; ++t) {
          // S = Q K^T (+ Q K_lo^T: plane 2 of the stage)
          const uint32_t kt = k_addr + t * 2 * C::K_BYTES;
#pragma unroll
          for (int k = 0; k < D / 16; ++k) {
            const uint32_t off = (k % 4) * 32;  // 16 K-elements within the 128-B row
            const uint64_t ad = umma_desc_sw128(q_addr + (k / 4) * (128 * 128) + off);
            const uint64_t bd = umma_desc_sw128(kt + (k / 4) * C::KV_HALF + off);
            umma_bf16(tmem + C::S_COL0 + b * kChunkKeys, ad, bd, idesc_s, (t | k) > 0 ? 1u : 0u);
          }
        }
        umma_commit(&s_full[b]);
        return true;
      };
      auto issue_pv = [&](int c) -> bool {
        const int st = c % kStages, b = c & 1;
        if (!mbar_wait(&p_full[b], (c >> 1) & 1, abort_flag)) return false;
        tc_fence_after();
        const uint32_t p_addr = smem_u32(sm + C::P_OFF + b * C::P_BYTES);
        const uint32_t v_addr = smem_u32(sm + C::KV_OFF + st * C::STAGE_BYTES + C::K_BYTES);
#pragma unroll
        for (int t = 0; t < TERMS; ++t) {
          // O += P V (+ P V_lo: plane 3 of the stage)
          const uint32_t vt = v_addr + t * 2 * C::K_BYTES;
#pragma unroll
          for (int k = 0; k < kChunkKeys / 16; ++k) {
            const uint64_t ad = umma_desc_sw128(p_addr + k * 32);
            // keys 16k..16k+15 = page k of the V plane; its d halves are C::PH_BYTES apart
            const uint64_t bd = umma_desc_sw128_mn(vt + k * C::PPL_BYTES, C::PH_BYTES, 1024);
            umma_bf16(tmem + C::O_COL, ad, bd, idesc_pv, (c > 0 || t > 0 || k > 0) ? 1u : 0u);
          }
        }
        umma_commit(&pv_done[b]);
        umma_commit(&kv_empty[st]);
        return true;
      };
      bool ok = true;
      if (nch > 0) ok = issue_s(0);
      for (int c = 0; ok && c < nch; ++c) {
        if (c + 1 < nch) ok = issue_s(c + 1);
        if (ok) ok = issue_pv(c);
      }
      if (!ok) {
        *abort_flag = 1;
        raise_status(p.status, DFLASH_ERR_TIMEOUT, 312);
      }
    }
  }

  // ------------------------------------------------ softmax (warps 0-3)
  const float sl2 = rsqrtf(static_cast<float>(D)) * 1.4426950408889634f;
  const int pair = dual ? warp / 2 : 0;                      // meaningful for warps < 4
  const int wip = dual ? warp % 2 : warp;                    // warp index within its pair
  const int row_l = wip * 32 + lane;                         // query row of this thread
  const bool active = warp < 4 && wip < n_act;
  const int c_step = dual ? 2 : 1;
  const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);
  float m_used = -INFINITY, l_sum = 0.f;
  bool sm_ok = true;
  if (active) {
    for (int c = pair; c < nch; c += c_step) {
      const int b = c & 1, st = c % kStages;
      // every wait's outcome is made warp-uniform: the tcgen05.ld/st below are
      // .sync.aligned and must be executed by all 32 lanes together
      if (!__all_sync(0xffffffffu, mbar_wait(&s_full[b], (c >> 1) & 1, abort_flag))) { sm_ok = false; break; }
      tc_fence_after();
      uint32_t sr0[32], sr1[32];
      tmem_ld32_nowait(lane_base + C::S_COL0 + b * kChunkKeys, sr0);
      tmem_ld32_nowait(lane_base + C::S_COL0 + b * kChunkKeys + 32, sr1);
      tmem_wait_ld(sr0);
      tmem_regs_ready(sr1);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_free[b]);
      int cntp[kChunkPages];
      bool full = true, stale = false;
#pragma unroll
      for (int pp = 0; pp < kChunkPages; ++pp) {
        cntp[pp] = pages_n[c * kChunkPages + pp];
        full &= (cntp[pp] == 16);
        stale |= (cntp[pp] > 0 && cntp[pp] < 16 && pages_s[c * kChunkPages + pp] >= 0);
      }
      float s[64];
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        s[j] = __uint_as_float(sr0[j]);
        s[32 + j] = __uint_as_float(sr1[j]);
      }
      uint32_t sv_addr = 0;  // FP8: the V scale of every key, folded into P
      if constexpr (FP8) {
        // K scales folded into the scores (S = scale_k * (q . codes))
        const uint32_t sk_addr = smem_u32(sm + C::SCB_OFF + st * C::SC_BYTES);
        sv_addr = sk_addr + kChunkKeys * 4;
#pragma unroll
        for (int j = 0; j < 64; j += 4) {
          const float4 k4 = ld_shared_f4(sk_addr + j * 4);
          s[j] *= k4.x;
          s[j + 1] *= k4.y;
          s[j + 2] *= k4.z;
          s[j + 3] *= k4.w;
        }
      }
      if (!full) {
        // invalid keys (stale or zero-filled rows) never contribute
#pragma unroll
        for (int j = 0; j < 64; ++j) s[j] = ((j % 16) < cntp[j / 16]) ? s[j] : -INFINITY;
      }
      if constexpr (CAUSAL) {
        // keys past this row's own position
        const int kpos0 = (pg_lo + c * kChunkPages) * 16;
        const int qpos = L + i0 + row_l / G;
        if (kpos0 + 63 > qpos) {
#pragma unroll
          for (int j = 0; j < 64; ++j) s[j] = (kpos0 + j <= qpos) ? s[j] : -INFINITY;
        }
      }
      float mx8[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) mx8[e] = fmaxf(s[e], s[e + 8]);
#pragma unroll
      for (int j = 16; j < 64; j += 8)
#pragma unroll
        for (int e = 0; e < 8; ++e) mx8[e] = fmaxf(mx8[e], s[j + e]);
      const float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                             fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
      const float mc = mx * sl2;
      // new reference maximum where the chunk's exceeds it by more than 2^8;
      // O and l of such rows are rescaled (warp-collective: lanes that keep
      // their maximum take alpha = 1)
      const bool raise_m = mc > m_used + kRescaleLog2;
      const bool rescale = raise_m && m_used != -INFINITY;
      if (__any_sync(0xffffffffu, rescale)) {
        if (!__all_sync(0xffffffffu, mbar_wait(&pv_done[(c - 1) & 1], ((c - 1) >> 1) & 1, abort_flag))) {
          sm_ok = false;
          break;
        }
        tc_fence_after();
        const float alpha = rescale ? ex2_approx(m_used - mc) : 1.f;
#pragma unroll 1
        for (int q = 0; q < D / 32; ++q) {
          uint32_t o[32];
          tmem_ld32_nowait(lane_base + C::O_COL + q * 32, o);
          tmem_wait_ld(o);
#pragma unroll
          for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
          tmem_st32(lane_base + C::O_COL + q * 32, o);
          tmem_wait_st();  // before o is reloaded
        }
        l_sum *= alpha;
      }
      if (raise_m) m_used = mc;
      // P = exp2(s*sl2 - m) in bf16 (masked keys: exp2(-inf) = 0)
      const float neg = (m_used == -INFINITY) ? 0.f : -m_used;
      uint32_t pk[32];
      float ls4[4] = {0.f, 0.f, 0.f, 0.f};
      float svv[FP8 ? 64 : 1];
      if constexpr (FP8) {
#pragma unroll
        for (int j = 0; j < 64; j += 4) {
          const float4 v4 = ld_shared_f4(sv_addr + j * 4);
          svv[j] = v4.x;
          svv[j + 1] = v4.y;
          svv[j + 2] = v4.z;
          svv[j + 3] = v4.w;
        }
      }
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const float p0 = ex2_approx(fmaf(s[2 * j], sl2, neg));
        const float p1 = ex2_approx(fmaf(s[2 * j + 1], sl2, neg));
        if constexpr (FP8)
          pk[j] = pack_bf16x2(p0 * svv[2 * j], p1 * svv[2 * j + 1]);  // P * scale_v
        else
          pk[j] = pack_bf16x2(p0, p1);
        ls4[j & 3] += p0 + p1;
      }
      l_sum += (ls4[0] + ls4[1]) + (ls4[2] + ls4[3]);
      // the P buffer b was last read by PV(c-2)
      if (c >= 2 && !__all_sync(0xffffffffu, mbar_wait(&pv_done[b], ((c - 2) >> 1) & 1, abort_flag))) {
        sm_ok = false;
        break;
      }
      uint8_t* pbuf = sm + C::P_OFF + b * C::P_BYTES;
      const int prow = warp * 32 + lane;  // MMA row = TMEM lane
#pragma unroll
      for (int c16 = 0; c16 < 8; ++c16)
        *reinterpret_cast<uint4*>(pbuf + swz128(prow, c16)) =
            make_uint4(pk[4 * c16], pk[4 * c16 + 1], pk[4 * c16 + 2], pk[4 * c16 + 3]);
      if (!FP8 && stale) {
        // rows past a context page's valid keys hold stale pool data: zero
        // their V rows (and low terms) so that 0 * V stays 0
        uint8_t* vst = sm + C::KV_OFF + st * C::STAGE_BYTES + C::K_BYTES;
        for (int idx = row_l; idx < kChunkKeys * C::HALVES * 8; idx += n_act * 32) {
          const int key = idx / (C::HALVES * 8), rem = idx % (C::HALVES * 8);
          const int hf = rem / 8, c16 = rem % 8;
          if ((key % 16) >= cntp[key / 16]) {
            uint8_t* v16 = vst + (key / 16) * C::PPL_BYTES + hf * C::PH_BYTES + swz128(key % 16, c16);
            *reinterpret_cast<uint4*>(v16) = make_uint4(0u, 0u, 0u, 0u);
            if (TERMS == 2) *reinterpret_cast<uint4*>(v16 + 2 * C::K_BYTES) = make_uint4(0u, 0u, 0u, 0u);
          }
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[b]);
    }
    if (!sm_ok) {
      *abort_flag = 1;
      if (lane == 0) raise_status(p.status, DFLASH_ERR_TIMEOUT, 313);
    }
    // the last PV of the CTA (it covers this pair's chunks too)
    if (sm_ok && nch > 0 &&
        !__all_sync(0xffffffffu, mbar_wait(&pv_done[(nch - 1) & 1], ((nch - 1) >> 1) & 1, abort_flag))) {
      *abort_flag = 1;
      if (lane == 0) raise_status(p.status, DFLASH_ERR_TIMEOUT, 314);
    }
  }

  // ------------------------------------------------ partials -> owning CTAs
  // With two warp pairs, the odd-chunk pair first hands its (O, m, l) to the
  // even-chunk pair through local shared memory (the Q/P area, free once the
  // last PV has completed), which merges the two states; one partial per row
  // and split then remains.  CTA q of the cluster merges query rows
  // [q*rpc, q*rpc + rpc): after the first cluster barrier every CTA's K/V
  // stages are free, and each row's partial is stored straight into the
  // owner's stage area (remote stores, no round trip); after the second
  // barrier the owner merges from its own shared memory.
  __syncthreads();
  tc_fence_after();
  const int SC = gridDim.x;
  const int n_part = 1;
  const int rpc = (R + SC - 1) / SC;
  constexpr int OS_LD = D + 4;  // padded row stride (floats): conflict-free row stores
  float* Xs = reinterpret_cast<float*>(sm + C::Q_OFF);       // [64][OS_LD] odd pair's O rows
  float* Xml = Xs + 64 * OS_LD;                               // [64][2]
  static_assert(64 * (D + 4) * 4 + 64 * 8 <= 2 * C::P_BYTES + C::Q_BYTES, "pair staging must fit Q/P");
  const bool have = active && __all_sync(0xffffffffu, nch > pair && !*abort_flag);
  if (dual && active && pair == 1) {  // warp-uniform
#pragma unroll 1
    for (int q = 0; q < D / 32; ++q) {
      uint32_t o[32];
      if (have) {
        tmem_ld32_nowait(lane_base + C::O_COL + q * 32, o);
        tmem_wait_ld(o);
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) o[j] = 0u;
      }
      float* dst = Xs + row_l * OS_LD + q * 32;
#pragma unroll
      for (int j = 0; j < 32; j += 4)
        *reinterpret_cast<uint4*>(dst + j) = make_uint4(o[j], o[j + 1], o[j + 2], o[j + 3]);
    }
    Xml[row_l * 2 + 0] = have ? m_used : -INFINITY;
    Xml[row_l * 2 + 1] = have ? l_sum : 0.f;
  }
  __syncthreads();
  float* Rb = reinterpret_cast<float*>(sm + C::KV_OFF);     // [rpc][SC][OS_LD]
  float* Rml = Rb + static_cast<size_t>(rpc) * n_part * SC * OS_LD;  // [rpc][SC][2]
  cluster_sync();
  tc_fence_after();
  if (active && pair == 0) {  // warp-uniform: the tcgen05.ld below needs all 32 lanes
    const bool mine = row_l < R;  // lanes past the real rows load but store nothing
    const int own = mine ? row_l / rpc : 0, lr = row_l % rpc;
    const int slot = lr * SC + split;
    const uint32_t dst = dsmem_map(smem_u32(Rb + static_cast<size_t>(slot) * OS_LD), own);
    // this pair's state and, with two pairs, the odd pair's
    float m0 = have ? m_used : -INFINITY, l0 = have ? l_sum : 0.f;
    float m1 = -INFINITY, l1 = 0.f;
    if (dual) {
      m1 = Xml[row_l * 2 + 0];
      l1 = Xml[row_l * 2 + 1];
    }
    const float mx = fmaxf(m0, m1);
    const float w0 = (m0 == -INFINITY) ? 0.f : exp2f(m0 - mx);
    const float w1 = (m1 == -INFINITY) ? 0.f : exp2f(m1 - mx);
#pragma unroll 1
    for (int q = 0; q < D / 32; ++q) {
      uint32_t o[32];
      if (have) {
        tmem_ld32_nowait(lane_base + C::O_COL + q * 32, o);
        tmem_wait_ld(o);
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) o[j] = 0u;
      }
      if (dual) {
        const float* x = Xs + row_l * OS_LD + q * 32;
#pragma unroll
        for (int j = 0; j < 32; ++j)
          o[j] = __float_as_uint(__uint_as_float(o[j]) * w0 + x[j] * w1);
      }
      if (mine) {
#pragma unroll
        for (int j = 0; j < 32; j += 4)
          asm volatile("st.shared::cluster.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst + (q * 32 + j) * 4),
                       "r"(o[j]), "r"(o[j + 1]), "r"(o[j + 2]), "r"(o[j + 3])
                       : "memory");
      }
    }
    if (mine) {
      const float mv = dual ? mx : m0, lv = dual ? l0 * w0 + l1 * w1 : l0;
      asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(
                       dsmem_map(smem_u32(Rml + static_cast<size_t>(slot) * 2), own)),
                   "f"(mv), "f"(lv)
                   : "memory");
    }
  }
  cluster_sync();

  // ------------------------------------------------ merge (local shared memory)
  {
    const int q = static_cast<int>(cluster_ctarank());
    constexpr int VEC = D / 32;  // floats per lane
    for (int lr = warp; lr < rpc && q * rpc + lr < R; lr += kThreads / 32) {
      const int r = q * rpc + lr;
      // lane pi = part * SC + split holds that partial's (m, l)
      float ms = -INFINITY, ls = 0.f;
      if (lane < n_part * SC) {
        const float2 v = *reinterpret_cast<const float2*>(Rml + (static_cast<size_t>(lr) * n_part * SC + lane) * 2);
        ms = v.x;
        ls = v.y;
      }
      const float mstar = warp_max(ms);
      const float w = (ms == -INFINITY) ? 0.f : exp2f(ms - mstar);
      const float lsum = warp_sum(w * ls);
      float acc[VEC];
#pragma unroll
      for (int e = 0; e < VEC; ++e) acc[e] = 0.f;
      const float* rb = Rb + static_cast<size_t>(lr) * n_part * SC * OS_LD + lane * VEC;
      for (int pi = 0; pi < n_part * SC; ++pi) {
        const float wp = __shfl_sync(0xffffffffu, w, pi);
        const float* src = rb + pi * OS_LD;
        if constexpr (VEC == 4) {
          const float4 v = *reinterpret_cast<const float4*>(src);
          acc[0] = fmaf(v.x, wp, acc[0]);
          acc[1] = fmaf(v.y, wp, acc[1]);
          acc[2] = fmaf(v.z, wp, acc[2]);
          acc[3] = fmaf(v.w, wp, acc[3]);
        } else {
          const float2 v = *reinterpret_cast<const float2*>(src);
          acc[0] = fmaf(v.x, wp, acc[0]);
          acc[1] = fmaf(v.y, wp, acc[1]);
        }
      }
      const float inv = 1.f / lsum;
      const int i = i0 + r / G, h = r % G;
      const size_t ob = ((static_cast<size_t>(req) * p.n + i) * p.hq + g * G + h) * D + lane * VEC;
#pragma unroll
      for (int e = 0; e < VEC; ++e) {
        const float v = acc[e] * inv;
        const uint16_t hi = f2bf(v);
        p.out[ob + e] = hi;
        if (p.out_lo != nullptr) p.out_lo[ob + e] = bf16_lo_part(v, hi);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 5) tmem_dealloc(tmem, C::TMEM_COLS);
}

template <int D, bool CAUSAL, int TERMS, bool FP8 = false>
cudaError_t launch_tc(const CUtensorMap* pool_map, const CUtensorMap* pool_v_map,
                      const CUtensorMap* kblk_map,
                      const CUtensorMap* vblk_map, const AttnTcParams& p, cudaStream_t s,
                      bool pdl) {
  using C = TcCfg<D, TERMS, FP8>;
  static thread_local int attr_device = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (attr_device != dev) {
    cudaError_t e = cudaFuncSetAttribute(attn_tc05_kernel<D, CAUSAL, TERMS, FP8>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(attn_tc05_kernel<D, CAUSAL, TERMS, FP8>,
                             cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    attr_device = dev;
  }
  cudaLaunchAttribute attrs[2];
  int na = 0;
  if (pdl) {
    attrs[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  attrs[na].id = cudaLaunchAttributeClusterDimension;
  attrs[na].val.clusterDim.x = p.n_splits;
  attrs[na].val.clusterDim.y = 1;
  attrs[na].val.clusterDim.z = 1;
  ++na;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.n_splits, p.batch * p.hkv, (p.n + p.rows_per_tile - 1) / p.rows_per_tile);
  cfg.blockDim = dim3(C::THREADS, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = s;
  cfg.attrs = attrs;
  cfg.numAttrs = na;
  count_launch();
  return cudaLaunchKernelEx(&cfg, attn_tc05_kernel<D, CAUSAL, TERMS, FP8>, *pool_map, *pool_v_map,
                            *kblk_map, *vblk_map, p);
}

}  // namespace

// Clusters of `cluster` CTAs (head_dim d) that can be resident at once.
// Cached per device (value + 1; 0 = not yet queried).  The queries run at
// model creation (attention_tc_prepare), outside any stream capture.
constexpr int kMaxDevices = 64;
static int g_active_clusters[kMaxDevices][2][kMaxAttnCluster + 1];

static int max_active_clusters(int d, int cluster) {
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= kMaxDevices) return 0;
  int& slot = g_active_clusters[dev][d == 128 ? 1 : 0][cluster];
  if (slot > 0) return slot - 1;
  const void* fn = d == 128 ? reinterpret_cast<const void*>(attn_tc05_kernel<128>)
                            : reinterpret_cast<const void*>(attn_tc05_kernel<64>);
  const int smem = d == 128 ? TcCfg<128>::SMEM : TcCfg<64>::SMEM;
  int n = 0;
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) == cudaSuccess &&
      cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cluster, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess) n = 0;
  }
  cudaGetLastError();
  slot = n + 1;
  return n;
}

void attention_tc_prepare(int d) {
  for (int c = 1; c <= kMaxAttnCluster; ++c) max_active_clusters(d, c);
}

// Pages per key split.  Every (request, KV head) pair is one cluster of
// splits; the estimate is the number of waves of resident clusters times one
// CTA's duration (a fixed cost per CTA plus a cost per 64-key chunk).
int attention_tc_split_pages(int d, int pairs, int total_pages) {
  constexpr double kFixUs = 5.0, kChunkUs = 0.8;
  double best = 1e30;
  int best_sp = (total_pages + kMaxAttnCluster - 1) / kMaxAttnCluster;
  for (int s = 1; s <= kMaxAttnCluster; ++s) {
    const int sp = (total_pages + s - 1) / s;
    if (sp > kMaxPagesTc) continue;
    const int splits = (total_pages + sp - 1) / sp;
    const int act = max_active_clusters(d, splits);
    if (act <= 0) continue;
    const double cta = kFixUs + ((sp + kChunkPages - 1) / kChunkPages) * kChunkUs;
    const double est = static_cast<double>((pairs + act - 1) / act) * cta;
    if (est < best * 0.999) {
      best = est;
      best_sp = sp;
    }
  }
  return best_sp;
}

bool attention_tc_ok(int d, int hq, int hkv, int n, int page_size, int split_pages) {
  return (d == 64 || d == 128) && page_size == 16 && hkv > 0 && hq % hkv == 0 &&
         n * (hq / hkv) <= 128 && split_pages <= kMaxPagesTc;
}

cudaError_t attention_tc_launch(const CUtensorMap* pool_map, const CUtensorMap* pool_v_map,
                                const CUtensorMap* kblk_map, const CUtensorMap* vblk_map,
                                const AttnTcParams& p, cudaStream_t s, bool pdl) {
  if (p.n_splits < 1 || p.n_splits > kMaxAttnCluster) return cudaErrorInvalidValue;
  if (p.rows_per_tile < 1 || p.rows_per_tile * (p.hq / p.hkv) > 128) return cudaErrorInvalidValue;
  if (p.causal) {
    // the target path: dual-state query tiles only, one- or two-term K/V
    if (p.rows_per_tile * (p.hq / p.hkv) > 64) return cudaErrorInvalidValue;
    if (p.kv_terms == 2) {
      if (p.d == 128) return launch_tc<128, true, 2>(pool_map, pool_v_map, kblk_map, vblk_map, p, s, pdl);
      if (p.d == 64) return launch_tc<64, true, 2>(pool_map, pool_v_map, kblk_map, vblk_map, p, s, pdl);
    } else {
      if (p.d == 128) return launch_tc<128, true, 1>(pool_map, pool_v_map, kblk_map, vblk_map, p, s, pdl);
      if (p.d == 64) return launch_tc<64, true, 1>(pool_map, pool_v_map, kblk_map, vblk_map, p, s, pdl);
    }
    return cudaErrorInvalidValue;
  }
  if (p.kv_terms == 2) return cudaErrorInvalidValue;
  if (p.fp8) {
    if (p.scales == nullptr) return cudaErrorInvalidValue;
    if (p.d == 128) return launch_tc<128, false, 1, true>(pool_map, pool_v_map, kblk_map, vblk_map, p, s, pdl);
    if (p.d == 64) return launch_tc<64, false, 1, true>(pool_map, pool_v_map, kblk_map, vblk_map, p, s, pdl);
    return cudaErrorInvalidValue;
  }
  if (p.d == 128) return launch_tc<128, false, 1>(pool_map, pool_v_map, kblk_map, vblk_map, p, s, pdl);
  if (p.d == 64) return launch_tc<64, false, 1>(pool_map, pool_v_map, kblk_map, vblk_map, p, s, pdl);
  return cudaErrorInvalidValue;
}

int attention_tc_target_split_pages() { return kTargetSplitPagesTc; }

}  // namespace dflash
