// Prefill and chunked-prefill rows (q_len > 1) of the step on tcgen05/TMEM, bf16.
//
// What it computes is the per-block pseudocode of "Continuous Batching"
// (languisher.top), section "Extension: the vLLM v1 implementation", for a
// request's query tile: context_len = seq_len - q_len, query token local_q
// attends kv_pos 0 .. context_len + local_q (or the last sliding_window of
// them), each resolved through block_table[req][kv_pos / BLOCK_SIZE]. The
// chunk's own tokens were scattered into the cache before this kernel runs
// (section "Extension: combining with chunked prefill": a chunk with a context
// continues a prompt already in the cache). Prefill is compute-bound
// ("Continuous batching mechanics", d9bl.com), so both products are dense
// contractions on the 5th-generation tensor cores:
//
// * Tile. One CTA owns 128 query rows = 128/G tokens x the G query heads of
//   one KV head (grouped-query packing: each K/V tile serves all G heads), and
//   walks the request's keys in tiles of 128 up to its causal bound. Only the
//   last tiles need the bound check; it is applied per row as a select.
// * Staging. The softmax threads copy their query rows into TMEM once; a TMA
//   warp loads each K and V tile page by page (a 4-D box per page through the block table, 128B
//   swizzle, one lane per page) into mbarrier rings (K: 4 stages, freed when S
//   is done; V: 3 stages, freed when PV is done); pages past the request read
//   as zeros.
// * Contraction. One thread issues S = Q K^T (M 128, N 128, K = head_dim; Q
//   from TMEM, K from swizzled shared memory, so only one operand streams
//   through shared memory) into a double-buffered TMEM accumulator,
//   and O += P V (M 128, N = head_dim, K 128) into a TMEM accumulator with P
//   read from TMEM where the softmax left it and V as the N-major
//   shared-memory operand. S of the next key tile is computed while the softmax
//   works on the current one.
// * Softmax. Four warps, one thread per row (= TMEM lane): load the S row with
//   tcgen05.ld, mask, exponentiate in base 2, write P (bf16 pairs, tcgen05.st)
//   into TMEM for the PV product. The running maximum is only raised (and O rescaled in TMEM)
//   when it grows by more than 2^8, which keeps every P <= 256 and the result
//   exact up to rounding. The last PV completes, O is divided by the row sum
//   and written out.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <float.h>

#include "common.cuh"
#include "launch.h"
#include "prefill.h"
#include "sm100_ptx.cuh"

namespace cb {

namespace {

constexpr int kRows = 128;             // query rows per tile
constexpr int kKeys = 128;             // keys per key tile
constexpr int kKStages = 4;            // K ring depth (K is free once S = Q K^T is done)
constexpr int kVStages = 3;            // V ring depth (V is free once O += P V is done)
constexpr int kThreads = 192;          // warps 0-3 softmax, 4 TMA, 5 MMA
constexpr float kRescaleLog2 = 8.f;    // raise the running max only when it grows by > 2^8
constexpr uint32_t kTmemCols = 512;    // S0: 0-127, S1: 128-255, O: 256-383, P: 384-447, Q: 448-511
constexpr uint32_t kTmemO = 256;
constexpr uint32_t kTmemP = 384;       // bf16 pairs: 128 keys in 64 columns
constexpr uint32_t kTmemQ = 448;       // bf16 pairs: head_dim <= 128 in 64 columns
constexpr int kHalfBytes = kRows * 128;  // 128 rows x 64 bf16 (one swizzle-atom column)

struct PfBars {
  uint64_t q_full;  // Q rows stored into TMEM by the four softmax warps
  uint64_t k_full[kKStages];
  uint64_t k_empty[kKStages];
  uint64_t v_full[kVStages];
  uint64_t v_empty[kVStages];
  uint64_t s_full[2];
  uint64_t s_free[2];
  uint64_t p_full;
  uint64_t o_done;
  uint64_t drain;
  uint32_t tmem_base;
};

struct Tile {
  int r, g, pair, qt;
  bool shadow;  // the odd last tile's partner: loads its half of K/V, stores nothing
};

// Cluster -> (request, KV head, pair of query tiles); entries are sorted
// heaviest first and each request's pairs are taken last first (the last has
// the most keys). CTA rank 0 of the cluster takes the pair's first tile.
CB_DEV Tile tile_of(const PrefillArgs& p, int cluster, int rank) {
  const int Hkv = p.a.num_kv_heads;
  int base = 0;
  for (int e = 0; e < p.n_entries; ++e) {
    const int nq = p.entries[e].n_qtiles;
    const int npairs = (nq + 1) / 2;
    const int n = npairs * Hkv;
    if (cluster < base + n) {
      const int k = cluster - base;
      Tile t;
      t.r = p.entries[e].r;
      t.g = k % Hkv;
      t.pair = npairs - 1 - k / Hkv;
      t.qt = 2 * t.pair + rank;
      t.shadow = t.qt >= nq;
      if (t.shadow) t.qt = nq - 1;
      return t;
    }
    base += n;
  }
  return Tile{-1, 0, 0, 0, true};
}

template <int D>
__host__ __device__ constexpr int kv_bytes() {
  return (D / 64) * kHalfBytes;
}

}  // namespace

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
prefill_tile_kernel(const __grid_constant__ CUtensorMap tmap_k,
                    const __grid_constant__ CUtensorMap tmap_v,
                    const __grid_constant__ PrefillArgs p) {
  static_assert(D == 64 || D == 128, "head_dim");
  constexpr int kHalves = D / 64;
  constexpr int kKV = kv_bytes<D>();
  extern __shared__ __align__(1024) uint8_t smem_dyn[];
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
  uint8_t* sK = base;
  uint8_t* sV = sK + kKStages * kKV;
  PfBars& bar = *reinterpret_cast<PfBars*>(sV + kVStages * kKV);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_cta_rank();  // clusters of two CTAs share K/V loads
  const Tile tile = tile_of(p, blockIdx.x / 2, (int)rank);
  if (tile.r < 0) return;  // uniform over the CTA, before any barrier

  if (threadIdx.x == 0) {
    mbar_init(&bar.q_full, 4);
    for (int s = 0; s < kKStages; ++s) {
      mbar_init(&bar.k_full[s], 1);
      mbar_init(&bar.k_empty[s], 2);  // released by both CTAs' S products
    }
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(&bar.v_full[s], 1);
      mbar_init(&bar.v_empty[s], 2);  // released by both CTAs' PV products
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bar.s_full[b], 1);
      mbar_init(&bar.s_free[b], 4);
    }
    mbar_init(&bar.p_full, 4);
    mbar_init(&bar.o_done, 1);
    mbar_init(&bar.drain, 1);
    fence_barrier_init();
  }
  if (warp == 4 && lane == 0) {
    prefetch_tensormap(&tmap_k);
    prefetch_tensormap(&tmap_v);
  }
  if (warp == 5) tmem_alloc(&bar.tmem_base, kTmemCols);
  grid_dependency_wait();  // the scatter of this step's K/V must be complete
  tcgen05_fence_before();
  cluster_sync();  // both CTAs' barriers exist before either multicasts into them
  tcgen05_fence_after();
  allow_dependent_launch();
  const uint32_t tmem = bar.tmem_base;

  // ---- request geometry
  const int r = tile.r;
  const int g = tile.g;
  const int q_start = __ldg(p.a.query_start_loc + r);
  const int q_len = __ldg(p.a.query_start_loc + r + 1) - q_start;
  const int seq = __ldg(p.a.seq_lens + r);
  const int ctx = seq - q_len;
  const int G = p.a.num_q_heads / p.a.num_kv_heads;
  const int TQ = p.tile_tokens;
  const int tok0 = tile.qt * TQ;
  const int tok_end = min(q_len, tok0 + TQ);
  // the cluster walks the union of its two tiles' key ranges
  const int pair_tok0 = 2 * tile.pair * TQ;
  const int pair_tok_end = min(q_len, pair_tok0 + 2 * TQ);
  const int W = p.a.sliding_window;
  const int first_key = W > 0 ? max(0, ctx + pair_tok0 - W + 1) : 0;
  const int last_key = min(ctx + pair_tok_end - 1, seq - 1);
  const int kt0 = first_key / kKeys;
  const int nkt = last_key / kKeys - kt0 + 1;
  bool ok = true;

  if (warp == 4) {
    // =================================================== TMA warp
    const int BS = p.a.block_size;
    const int box = p.box_keys;
    const int ppt = kKeys / box;  // pages per key tile
    const int npages_req = (seq + BS - 1) / BS;
    const int32_t* bt = p.a.block_table + (long long)r * p.a.bt_stride;
    // page ids of key tile j (lane i < ppt: page i of the tile)
    auto tile_pages = [&](int j) -> int {
      const int lp = (kt0 + j) * kKeys / BS + lane;
      int pg = p.a.num_blocks;  // past the pool: the TMA fills zeros
      if (lane < ppt && lp < npages_req) {
        pg = __ldg(bt + lp);
        if (pg < 0 || pg >= p.a.num_blocks) {
          record_error(p.a.error_word, 0x1);
          pg = p.a.num_blocks;
        }
      }
      return pg;
    };
    // one tensor's key tile j into `dst` of both CTAs: the tile's boxes (ppt
    // pages x kHalves halves) are split between the two CTAs, each box
    // multicast to both; lane i issues box 2i + rank (lanes issue in parallel)
    const int nbox = ppt * kHalves;
    auto issue_tile = [&](int j, int pg, const CUtensorMap* map, uint8_t* dst, uint64_t* full) {
      const int key0 = BS > kKeys ? ((kt0 + j) * kKeys) % BS : 0;
      const int bx = 2 * lane + (int)rank;
      const int page = bx / kHalves;
      const int half = bx % kHalves;
      const int pgb = __shfl_sync(0xffffffffu, pg, page & 31);
      __syncwarp();  // the expect_tx above is registered first
      if (bx < nbox)
        tma_load_4d_multicast(dst + half * kHalfBytes + page * box * 128, map, full, half * 64,
                              key0, g, pgb, (uint16_t)0x3);
    };
    // K runs one tile ahead of V; page ids are read one tile ahead
    int k_issued = 0, v_issued = 0;
    int ids_next = tile_pages(0);
    int ids_v = 0;
    for (int j = -1; j < nkt && ok; ++j) {
      const int jk = j + 1;
      const int ids_k = ids_next;
      if (jk + 1 < nkt) ids_next = tile_pages(jk + 1);
      if (jk < nkt) {
        const int s = jk % kKStages;
        if (jk >= kKStages &&
            !mbar_wait_warp(&bar.k_empty[s], (uint32_t)(((jk / kKStages) - 1) & 1))) {
          ok = false;
          break;
        }
        if (lane == 0) mbar_arrive_expect_tx(&bar.k_full[s], (uint32_t)kKV);
        issue_tile(jk, ids_k, &tmap_k, sK + s * kKV, &bar.k_full[s]);
        k_issued = jk + 1;
      }
      if (j >= 0) {
        const int s = j % kVStages;
        if (j >= kVStages &&
            !mbar_wait_warp(&bar.v_empty[s], (uint32_t)(((j / kVStages) - 1) & 1))) {
          ok = false;
          break;
        }
        if (lane == 0) mbar_arrive_expect_tx(&bar.v_full[s], (uint32_t)kKV);
        issue_tile(j, ids_v, &tmap_v, sV + s * kKV, &bar.v_full[s]);
        v_issued = j + 1;
      }
      __syncwarp();
      ids_v = ids_k;
    }
    if (!ok && lane == 0) {
      record_error(p.a.error_word, 0x4);
      // the copies already issued land before the CTA's shared memory is released
      for (int jj = k_issued > kKStages ? k_issued - kKStages : 0; jj < k_issued; ++jj)
        mbar_wait(&bar.k_full[jj % kKStages], (uint32_t)((jj / kKStages) & 1));
      for (int jj = v_issued > kVStages ? v_issued - kVStages : 0; jj < v_issued; ++jj)
        mbar_wait(&bar.v_full[jj % kVStages], (uint32_t)((jj / kVStages) & 1));
    }
  } else if (warp == 5) {
    // =================================================== MMA issuer
    if (lane == 0) {
      constexpr uint32_t idS = umma_idesc_bf16(kRows, kKeys, false);
      constexpr uint32_t idO = umma_idesc_bf16(kRows, D, true);
      if (!mbar_wait(&bar.q_full, 0)) ok = false;
      for (int j = 0; j <= nkt && ok; ++j) {
        if (j < nkt) {
          // S_j = Q K_j^T into S buffer j % 2
          const int sb = j & 1;
          const int s = j % kKStages;
          if (j >= 2 && !mbar_wait(&bar.s_free[sb], (uint32_t)(((j >> 1) - 1) & 1))) {
            ok = false;
            break;
          }
          if (!mbar_wait(&bar.k_full[s], (uint32_t)((j / kKStages) & 1))) {
            ok = false;
            break;
          }
          tcgen05_fence_after();
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {
            const uint32_t ka = smem_u32(sK + s * kKV) + (ks >> 2) * kHalfBytes + (ks & 3) * 32;
            umma_bf16_tmem_a(tmem + sb * kKeys, tmem + kTmemQ + ks * 8,
                             umma_desc_sw128(ka, 16, 1024), idS, ks > 0);
          }
          umma_commit(&bar.s_full[sb]);
          umma_commit_multicast(&bar.k_empty[s], (uint16_t)0x3);
        }
        if (j >= 1) {
          // O += P_{j-1} V_{j-1}
          const int jj = j - 1;
          const int s = jj % kVStages;
          if (!mbar_wait(&bar.p_full, (uint32_t)(jj & 1)) ||
              !mbar_wait(&bar.v_full[s], (uint32_t)((jj / kVStages) & 1))) {
            ok = false;
            break;
          }
          tcgen05_fence_after();
#pragma unroll
          for (int ks = 0; ks < kKeys / 16; ++ks) {
            const uint32_t va = smem_u32(sV + s * kKV) + ks * 2048;
            umma_bf16_tmem_a(tmem + kTmemO, tmem + kTmemP + ks * 8,
                             umma_desc_sw128(va, kHalfBytes, 1024), idO,
                             (jj > 0 || ks > 0) ? 1u : 0u);
          }
          umma_commit(&bar.o_done);
          umma_commit_multicast(&bar.v_empty[s], (uint16_t)0x3);
        }
      }
      if (!ok) record_error(p.a.error_word, 0x4);
      // every MMA this thread issued has completed before the TMEM is released
      umma_commit(&bar.drain);
      mbar_wait(&bar.drain, 0);
    }
    __syncwarp();
  } else {
    // =================================================== softmax warps
    const int row = threadIdx.x;  // TMEM lane = tile row
    const uint32_t lane_addr = (uint32_t)(warp * 32) << 16;
    const int tok = tok0 + row / G;
    const int hh = row % G;
    const bool row_valid = tok < q_len && !tile.shadow;
    const int qpos = ctx + tok;
    const int max_kv = min(qpos, seq - 1);
    const int min_kv = W > 0 ? max(0, qpos - W + 1) : 0;
    const float sl2 = p.a.scale_log2;
    // keys every row of the tile attends: [tile_min_kv_max, tile_max_kv_min]
    const int tile_max_kv_min = min(ctx + tok0, seq - 1);
    const int tile_min_kv_max = W > 0 ? max(0, ctx + tok_end - 1 - W + 1) : 0;
    // this row's query (one token, one head: head_dim contiguous bf16) into TMEM as
    // the A operand of S = Q K^T; rows past the step read as zeros
    {
      const long long qrow = (long long)q_start + tok;
      const uint4* src = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.a.q) +
                                                        (qrow * p.a.num_q_heads + g * G + hh) * D);
      const bool in_step = qrow < p.a.num_tokens;
#pragma unroll
      for (int c0 = 0; c0 < D / 2; c0 += 16) {
        uint32_t qk[16];
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const uint4 x = in_step ? __ldg(src + c0 / 4 + v) : make_uint4(0, 0, 0, 0);
          qk[4 * v + 0] = x.x;
          qk[4 * v + 1] = x.y;
          qk[4 * v + 2] = x.z;
          qk[4 * v + 3] = x.w;
        }
        tmem_st16(tmem + lane_addr + kTmemQ + c0, qk);
      }
      tmem_wait_st();
      tcgen05_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar.q_full);
    }
    float m_ref = -FLT_MAX;
    float l = 0.f;
    for (int j = 0; j < nkt; ++j) {
      const int kt = kt0 + j;
      const int sb = j & 1;
      if (!mbar_wait_warp(&bar.s_full[sb], (uint32_t)((j >> 1) & 1))) {
        ok = false;
        break;
      }
      tcgen05_fence_after();
      uint32_t sr[kKeys];
#pragma unroll
      for (int c0 = 0; c0 < kKeys; c0 += 32)
        tmem_ld32(tmem + lane_addr + sb * kKeys + c0, *reinterpret_cast<uint32_t(*)[32]>(sr + c0));
      tmem_wait_ld();
      float* sv = reinterpret_cast<float*>(sr);
      tcgen05_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar.s_free[sb]);
      // mask (bounds only; tiles inside every row's range need none) and row
      // maximum of the raw scores (the scale is positive, so it commutes with max)
      const int key_base = kt * kKeys;
      if (key_base < tile_min_kv_max || key_base + kKeys - 1 > tile_max_kv_min) {
#pragma unroll
        for (int c = 0; c < kKeys; ++c) {
          const int key = key_base + c;
          if (key < min_kv || key > max_kv) sv[c] = -INFINITY;
        }
      }
      float mx8[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) mx8[k] = sv[k];
#pragma unroll
      for (int c = 8; c < kKeys; ++c) mx8[c & 7] = fmaxf(mx8[c & 7], sv[c]);
      const float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                             fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7]))) * sl2;
      const bool need = mx > m_ref + kRescaleLog2;
      const float alpha = need ? ex2_approx(m_ref - mx) : 1.f;
      if (need) m_ref = mx;
      // p = 2^(s * scale_log2 - m): one FFMA and one SFU op per score
      float sum8[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) sum8[k] = 0.f;
#pragma unroll
      for (int c = 0; c < kKeys; ++c) {
        sv[c] = ex2_approx(fmaf(sv[c], sl2, -m_ref));
        sum8[c & 7] += sv[c];
      }
      const float sum = ((sum8[0] + sum8[1]) + (sum8[2] + sum8[3])) +
                        ((sum8[4] + sum8[5]) + (sum8[6] + sum8[7]));
      l = l * alpha + sum;
      // P and O belong to the previous PV product until it completes
      if (j >= 1) {
        if (!mbar_wait_warp(&bar.o_done, (uint32_t)((j - 1) & 1))) {
          ok = false;
          break;
        }
        tcgen05_fence_after();
        if (__any_sync(0xffffffffu, need)) {
#pragma unroll
          for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t o32[32];
            tmem_ld32(tmem + lane_addr + kTmemO + c0, o32);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) o32[i] = __float_as_uint(__uint_as_float(o32[i]) * alpha);
            tmem_st32(tmem + lane_addr + kTmemO + c0, o32);
          }
          tmem_wait_st();
        }
      }
      // P row as bf16 pairs into TMEM (lane = row), the A operand of the PV product
#pragma unroll
      for (int c0 = 0; c0 < kKeys; c0 += 32) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) pk[i] = pack_bf16x2(sv[c0 + 2 * i], sv[c0 + 2 * i + 1]);
        tmem_st16(tmem + lane_addr + kTmemP + c0 / 2, pk);
      }
      // V rows past the end of the sequence hold unrelated data: zero them so
      // that 0 * V cannot produce a NaN (row index = key index in the tile)
      if (key_base + kKeys > seq) {
        if (!mbar_wait_warp(&bar.v_full[j % kVStages], (uint32_t)((j / kVStages) & 1))) {
          ok = false;
          break;
        }
        if (key_base + row >= seq) {
#pragma unroll
          for (int h = 0; h < kHalves; ++h)
#pragma unroll
            for (int c = 0; c < 8; ++c)
              *reinterpret_cast<uint4*>(sV + (j % kVStages) * kKV + h * kHalfBytes + row * 128 + c * 16) =
                  make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
      }
      tmem_wait_st();
      tcgen05_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar.p_full);
    }
    // ---- epilogue: O / l for the rows of this tile
    if (ok && !mbar_wait_warp(&bar.o_done, (uint32_t)((nkt - 1) & 1))) ok = false;
    if (ok) {
      tcgen05_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(p.a.out) +
                            ((long long)(q_start + tok) * p.a.num_q_heads + g * G + hh) * D;
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t o32[32];
        tmem_ld32(tmem + lane_addr + kTmemO + c0, o32);
        tmem_wait_ld();
        if (row_valid) {
#pragma unroll
          for (int c8 = 0; c8 < 4; ++c8) {
            uint4 v;
            v.x = pack_bf16x2(__uint_as_float(o32[c8 * 8 + 0]) * inv, __uint_as_float(o32[c8 * 8 + 1]) * inv);
            v.y = pack_bf16x2(__uint_as_float(o32[c8 * 8 + 2]) * inv, __uint_as_float(o32[c8 * 8 + 3]) * inv);
            v.z = pack_bf16x2(__uint_as_float(o32[c8 * 8 + 4]) * inv, __uint_as_float(o32[c8 * 8 + 5]) * inv);
            v.w = pack_bf16x2(__uint_as_float(o32[c8 * 8 + 6]) * inv, __uint_as_float(o32[c8 * 8 + 7]) * inv);
            *reinterpret_cast<uint4*>(orow + c0 + c8 * 8) = v;
          }
        }
      }
    } else if (lane == 0) {
      record_error(p.a.error_word, 0x4);
    }
  }

  // ---- teardown: every tcgen05 access is complete before the columns are
  // freed, and neither CTA leaves while the other may still write into it
  tcgen05_fence_before();
  __syncthreads();
  cluster_sync();
  if (warp == 5) {
    tcgen05_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ------------------------------------------------------------------ host

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

cudaError_t encode(CUtensorMap* map, void* ptr, int rank, const cuuint64_t* dims,
                   const cuuint64_t* strides, const cuuint32_t* box) {
  auto fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, ptr, dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int D>
cudaError_t launch_d(const PrefillArgs& p, cudaStream_t s) {
  const StepArgs& a = p.a;
  const cuuint64_t e = 2;
  CUtensorMap mk, mv;
  cudaError_t err = cudaSuccess;
  // caches as (d, key in page, head, page); box: 64 of d, box_keys keys, one head, one page
  cuuint64_t cd[4] = {(cuuint64_t)D, (cuuint64_t)a.block_size, (cuuint64_t)a.num_kv_heads,
                      (cuuint64_t)a.num_blocks};
  cuuint64_t cs[3] = {(cuuint64_t)a.num_kv_heads * D * e, (cuuint64_t)D * e,
                      (cuuint64_t)a.block_size * a.num_kv_heads * D * e};
  cuuint32_t cb_[4] = {64, (cuuint32_t)p.box_keys, 1, 1};
  err = encode(&mk, a.k_cache, 4, cd, cs, cb_);
  if (err == cudaSuccess) err = encode(&mv, a.v_cache, 4, cd, cs, cb_);
  if (err != cudaSuccess) return err;
  auto kern = prefill_tile_kernel<D>;
  static bool attr_set = false;
  const size_t smem = prefill_smem_bytes(D);
  if (!attr_set) {
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    attr_set = true;
  }
  return launch_pdl_cluster(kPrefillTc, kern, dim3(p.total_ctas), dim3(kThreads), 2, smem, s, mk, mv,
                            p);
}

}  // namespace

size_t prefill_smem_bytes(int head_dim) {
  const size_t kv = (size_t)(head_dim / 64) * kHalfBytes;
  size_t b = 1024 + (kKStages + kVStages) * kv + sizeof(PfBars);
  // at least ~half the SM's shared memory, so that a second CTA (and a second
  // 512-column TMEM allocation) never lands on the same SM
  if (b < 120 * 1024) b = 120 * 1024;
  return b;
}

cudaError_t launch_prefill(const PrefillArgs& p, cudaStream_t stream) {
  if (p.total_ctas <= 0) return cudaSuccess;
  if (p.a.head_dim == 64) return launch_d<64>(p, stream);
  return launch_d<128>(p, stream);
}

}  // namespace cb
