// Prefill and chunked-prefill rows (q_len > 1) of the step on tcgen05/TMEM, bf16.
//
// What it computes is the per-block pseudocode of "Continuous Batching"
// (languisher.top), section "Extension: the vLLM v1 implementation", for a
// request's query tile: context_len = seq_len - q_len, query token local_q
// attends kv_pos 0 .. context_len + local_q (or the last sliding_window of
// them), each resolved through block_table[req][kv_pos / BLOCK_SIZE]. The
// chunk's own tokens are this step's new K/V rows (section "Extension: combining
// with chunked prefill": a chunk with a context continues a prompt already in the
// cache). Prefill is compute-bound
// ("Continuous batching mechanics", d9bl.com), so both products are dense
// contractions on the 5th-generation tensor cores:
//
// * Tiles. A query tile is 128 rows = 128/G tokens x the G query heads of one
//   KV head (grouped-query packing: each K/V tile serves all G heads). A unit of
//   work is two consecutive query tiles A and B of a request for one KV head; its
//   key range (the union of the two tiles') is walked in tiles of 128 keys, so
//   each K/V tile loaded serves 256 rows. Only the tiles at a bound need the
//   per-row causal or window check.
// * Persistent CTAs. One CTA per SM (at most one per unit) claims units from the
//   step's list, heaviest first, through an atomic counter in the workspace, and
//   passes each to its roles through a two-slot ring in shared memory; the next
//   unit's query tiles and first K/V tiles load while the current one finishes.
// * Staging. The K TMA warp loads each unit's two query tiles (a 3-D box of the
//   G heads x TQ tokens per half of head_dim). Two TMA warps load the K and the V
//   tiles page by page (a 4-D box per page and 64-wide half of head_dim through
//   the block table, 128B swizzle, one lane per box) into one mbarrier ring in
//   the order K0, V0, K1, V1, ...; pages past the request read as zeros. The
//   step's own new positions are read from k_new / v_new where their slot is
//   their own; the softmax warps of CTAs with no unit left copy the new rows into
//   the cache.
// * Contraction. One MMA warp issues, for key tile j,
//     O_A += P_A V_j,  S_A = Q_A K_{j+1}^T,  O_B += P_B V_j,  S_B = Q_B K_{j+1}^T
//   (M 128; N head_dim or 128; K in steps of 16), accumulating in TMEM, whose
//   512 columns hold S_A, S_B, O_A, O_B. The softmax writes P (bf16 pairs)
//   over the first half of its own S columns, and PV reads it from there as
//   the TMEM A operand. One thread's MMAs execute in issue order, so S_{j+1}
//   overwrites P_j only after PV_j has read it, and the completion of S_{j+1}
//   also tells the softmax that PV_j no longer uses O. The fixed order
//   alternates the two groups, so each group's next S follows its P at once.
// * Softmax. Two warpgroups, one per query tile, one thread per row (= TMEM
//   lane): load the S row with tcgen05.ld, mask at the bounds, exponentiate in
//   base 2, store P with tcgen05.st. While one group works on its tile, the
//   tensor pipe runs the other group's products, so exponentials and MMAs
//   overlap. The running maximum is only raised (and O rescaled in TMEM) when
//   it grows by more than 2^8, which keeps every P <= 256 and the result exact
//   up to rounding. After the last PV, O is divided by the row sum and written
//   in whole 128-byte lines (32-byte pieces transposed within groups of four lanes).
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
constexpr int kTiles = 2;              // query tiles per CTA, one softmax warpgroup each
constexpr int kSoftmaxThreads = kTiles * kRows;
constexpr int kWarpTma = kSoftmaxThreads / 32;
constexpr int kWarpMma = kWarpTma + 1;
constexpr int kWarpTmaV = kWarpMma + 1;  // kWarpTma loads K tiles, kWarpTmaV V tiles
// The fourth warp of the last warpgroup (warp 11) has no role: setmaxnreg is executed per
// warpgroup, so the group of the TMA and MMA warps is complete.
constexpr int kThreads = kSoftmaxThreads + 128;
// Registers: 384 threads launch with 168 each (64,512 of the SM's 65,536); a thread's S
// row alone is 128 of them. The TMA and MMA warpgroup then gives back registers down to
// kRegsIssue each and the softmax warpgroups take kRegsSoftmax each. The roles share no
// code after the split, so the compiler allocates each within its own budget (with one
// budget for the whole kernel the softmax loop spilled).
constexpr int kThreadsBound = kThreads;
constexpr int kRegsLaunch = 168;
constexpr int kRegsIssue = 120;
constexpr int kRegsSoftmax = 192;
static_assert(kRegsIssue * 128 + kRegsSoftmax * kSoftmaxThreads <= kRegsLaunch * kThreads,
              "an increase waits for registers the launch does not hold");
constexpr float kRescaleLog2 = 8.f;    // raise the running max only when it grows by > 2^8
constexpr uint32_t kTmemCols = 512;    // S_A 0-127, S_B 128-255, O_A, O_B from 256 (head_dim each)
constexpr int kHalfBytes = kRows * 128;  // 128 rows x 64 bf16: one swizzle-atom column of a tile
constexpr int kMaxStages = 8;

// Bytes of one Q, K or V tile (128 rows x head_dim bf16).
template <int D>
__host__ __device__ constexpr int tile_bytes() {
  return (D / 64) * kHalfBytes;
}

// A unit of work: query tiles 2 pair and 2 pair + 1 of request r, KV head g (live = 0:
// no more units).
struct UnitDesc {
  int r, q_start, q_len, seq_len, g, pair, live;
};

// Geometry of a unit (request, KV head g, pair of query tiles): the union of the two
// tiles' key ranges is walked in key tiles kt0 .. kt0 + nkt - 1.
struct Geo {
  int r, g, q_start, q_len, seq, ctx, qt0, has_b, tok0, tok_end, kt0, nkt;
};

CB_DEV Geo geo_of(int r, int q_start, int q_len, int seq_len, int g, int pair, int TQ, int W) {
  Geo e;
  e.r = r;
  e.g = g;
  e.q_start = q_start;
  e.q_len = q_len;
  e.seq = seq_len;
  e.ctx = seq_len - q_len;
  e.qt0 = kTiles * pair;
  e.has_b = e.qt0 + 1 < (q_len + TQ - 1) / TQ;
  e.tok0 = e.qt0 * TQ;
  e.tok_end = min(q_len, e.tok0 + kTiles * TQ);
  const int first_key = W > 0 ? max(0, e.ctx + e.tok0 - W + 1) : 0;
  const int last_key = min(e.ctx + e.tok_end - 1, e.seq - 1);
  e.kt0 = first_key / kKeys;
  e.nkt = last_key / kKeys - e.kt0 + 1;
  return e;
}

CB_DEV Geo geo_of(const UnitDesc& d, int TQ, int W) {
  return geo_of(d.r, d.q_start, d.q_len, d.seq_len, d.g, d.pair, TQ, W);
}

// Warps that read the unit ring (the V TMA warp, the MMA warp, eight softmax warps).
constexpr int kUnitReaders = 2 + kSoftmaxThreads / 32;

struct PfBars {
  uint64_t q_full;              // both tiles' query rows in shared memory (tensor copies)
  uint64_t q_empty;             // the unit's last S products are done (query buffer free)
  uint64_t full[kMaxStages];    // ring slot loaded (K0, V0, K1, V1, ...)
  uint64_t empty[kMaxStages];   // ring slot released by the MMAs that read it
  uint64_t s_full[kTiles];      // S_t in TMEM (and the PV product before it complete)
  uint64_t p_full[kTiles];      // P_t in TMEM (the group's four warps)
  uint64_t o_done[kTiles];      // O_t final (its last PV product complete)
  uint64_t o_free[kTiles];      // O_t read by the epilogue (the group's four warps)
  uint64_t unit_full[2];        // unit ring slot written (the scheduler)
  uint64_t unit_empty[2];       // unit ring slot read (every other warp)
  UnitDesc unit[2];
  uint64_t drain;
  uint64_t never;               // nothing arrives here: the test hook's wait on it runs out
  uint32_t tmem_base;
  int abort;                    // a wait gave up: the other roles stop waiting
  int issued[kMaxStages];       // ring index of the latest copy issued into each slot
  int q_loads;                  // query-tile copies issued so far
};

// Ring depth: the shared memory left after the two query tiles, the barriers
// and the alignment slack, at most kMaxStages tiles.
template <int D>
__host__ __device__ constexpr int ring_stages() {
  return (kPrefillSmemLimit - 1024 - (int)sizeof(PfBars) - kTiles * tile_bytes<D>()) / tile_bytes<D>() > kMaxStages
             ? kMaxStages
             : (kPrefillSmemLimit - 1024 - (int)sizeof(PfBars) - kTiles * tile_bytes<D>()) / tile_bytes<D>();
}

template <int D>
__host__ __device__ constexpr size_t smem_bytes() {
  return 1024 + (size_t)(kTiles + ring_stages<D>()) * tile_bytes<D>() + sizeof(PfBars);
}

struct Work {
  int e, g, pair;
};

// Unit index of the step's list -> (entry, KV head, pair of query tiles); entries are
// sorted heaviest first and each request's pairs are taken last first (the last has the
// most keys), so the list runs heaviest first.
CB_DEV Work work_of(const PrefillArgs& p, int cta) {
  const int Hkv = p.a.num_kv_heads;
  int base = 0;
  for (int e = 0; e < p.n_entries; ++e) {
    const int npairs = (p.entries[e].n_qtiles + 1) / 2;
    const int n = npairs * Hkv;
    if (cta < base + n) {
      const int k = cta - base;
      return Work{e, k % Hkv, npairs - 1 - k / Hkv};
    }
    base += n;
  }
  return Work{-1, 0, 0};
}

// The pages of key tile `key_base` in `gen` (bit i: page i of the tile), row by row into
// the ring slot `dst` (128B-swizzled rows of 64 of head_dim per half): a new position whose
// slot is its own (bit clear in `bad`) from the step's new rows, any other from its cache
// page; positions past the request as zeros. Out of line: the path is rare (pages that
// straddle the context end or hold a foreign slot), and kept inline its registers and code
// slowed the TMA warps' common path (~3% of a long unit's key loop).
template <int D>
__device__ __noinline__ void copy_rows(uint8_t* dst, unsigned gen, int ids_cur, unsigned bad0,
                                       unsigned bad1, unsigned bad2, unsigned bad3, int key_base, int ctx, int seq, int q_start, int g, int Hkv,
                                       int BS, int box, const uint4* new_rows, const uint4* cache,
                                       int num_blocks, int32_t* error_word) {
  constexpr int kHalves = D / 64;
  constexpr int kBatch = 4;  // 16-byte chunks e = lane + 32 m of (row, half, chunk), loads first
  const int lane = threadIdx.x & 31;
  const int bs_mask = BS - 1;
  for (unsigned m = gen; m != 0u; m &= m - 1u) {
    const int pi = __ffs(m) - 1;
    const int pg = __shfl_sync(0xffffffffu, ids_cur, pi);
    const int kpi = key_base + pi * box;
    const bool pg_ok = pg >= 0 && pg < num_blocks;
    const int nchunks = box * kHalves * 8;
    for (int e0 = 0; e0 < nchunks; e0 += 32 * kBatch) {
      uint4 v[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int e = e0 + lane + 32 * u;
        const int row = e / (kHalves * 8), h = (e / 8) % kHalves, c = e % 8;
        const int pos = kpi + row;
        v[u] = make_uint4(0u, 0u, 0u, 0u);
        if (e < nchunks && pos < seq) {
          const int kk = pos - key_base;
          const unsigned bw = kk < 32 ? bad0 : kk < 64 ? bad1 : kk < 96 ? bad2 : bad3;
          const bool own = pos >= ctx && ((bw >> (kk & 31)) & 1u) == 0u;
          if (own) {
            v[u] = __ldg(new_rows + (((long long)(q_start + pos - ctx) * Hkv + g) * D + h * 64) / 8 + c);
          } else if (pg_ok) {
            v[u] = __ldg(cache + (((long long)pg * BS + (pos & bs_mask)) * Hkv + g) * (D / 8) + h * 8 + c);
          } else if (c == 0 && h == 0) {
            record_error(error_word, 0x1);
          }
        }
      }
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int e = e0 + lane + 32 * u;
        const int row = e / (kHalves * 8), h = (e / 8) % kHalves, c = e % 8;
        const int trow = pi * box + row;  // row within the tile
        if (e < nchunks)
          *reinterpret_cast<uint4*>(dst + h * kHalfBytes + trow * 128 + ((c ^ (trow & 7)) << 4)) = v[u];
      }
    }
  }
}

}  // namespace

template <int D>
__global__ void __launch_bounds__(kThreadsBound, 1)
prefill_tile_kernel(const __grid_constant__ CUtensorMap tmap_k,
                    const __grid_constant__ CUtensorMap tmap_v,
                    const __grid_constant__ CUtensorMap tmap_kn,
                    const __grid_constant__ CUtensorMap tmap_vn,
                    const __grid_constant__ CUtensorMap tmap_q,
                    const __grid_constant__ PrefillArgs p) {
  static_assert(D == 64 || D == 128, "head_dim");
  constexpr int kHalves = D / 64;
  constexpr int kTile = tile_bytes<D>();
  constexpr int kStages = ring_stages<D>();
  static_assert(kStages >= 3, "ring depth");
  static_assert(smem_bytes<D>() <= (size_t)kPrefillSmemLimit, "shared memory");
  extern __shared__ __align__(1024) uint8_t smem_dyn[];
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = base;
  uint8_t* sRing = sQ + kTiles * kTile;
  PfBars& bar = *reinterpret_cast<PfBars*>(sRing + kStages * kTile);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int Hkv = p.a.num_kv_heads;
  const int G = p.a.num_q_heads / Hkv;  // divides 128 (the launch checks): a power of two
  const int TQ = p.tile_tokens;
  const int W = p.a.sliding_window;
  // Graph replays: the one unit of this CTA, found with a block scan over the device
  // metadata (request order; each request with q_len > 1 has ceil(n_qtiles / 2) * Hkv).
  __shared__ UnitDesc s_first;  // the unit found on the device (kept out of registers)
  if (p.device_work) {
    grid_dependency_wait();
    __shared__ int s_tot[kThreads / 32];
    __shared__ int s_hit[2];
    if (threadIdx.x == 0) s_hit[0] = -1;
    int carry = 0;
    for (int base_r = 0; base_r < p.a.num_requests; base_r += kThreads) {
      const int rr = base_r + threadIdx.x;
      int n = 0;
      if (rr < p.a.num_requests) {
        const int ql = __ldg(p.a.query_start_loc + rr + 1) - __ldg(p.a.query_start_loc + rr);
        if (ql > 1) n = ((ql + TQ - 1) / TQ + 1) / 2 * Hkv;
      }
      int v = n;  // inclusive warp scan
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += y;
      }
      if (lane == 31) s_tot[warp] = v;
      __syncthreads();
      int before = carry;
      for (int k = 0; k < warp; ++k) before += s_tot[k];
      const int incl = before + v;
      if (n > 0 && incl - n <= (int)blockIdx.x && (int)blockIdx.x < incl) {
        s_hit[0] = rr;
        s_hit[1] = (int)blockIdx.x - (incl - n);
      }
      for (int k = 0; k < kThreads / 32; ++k) carry += s_tot[k];
      __syncthreads();
      if (s_hit[0] >= 0) break;
    }
    if (s_hit[0] < 0) return;  // past the step's work: uniform over the CTA
    const int rr = s_hit[0];
    const int k = s_hit[1];
    const int qs0 = __ldg(p.a.query_start_loc + rr);
    const int ql = __ldg(p.a.query_start_loc + rr + 1) - qs0;
    const int npairs = ((ql + TQ - 1) / TQ + 1) / 2;
    if (threadIdx.x == 0)
      s_first = UnitDesc{rr, qs0, ql, __ldg(p.a.seq_lens + rr), k % Hkv, npairs - 1 - k / Hkv, 1};
  }

  if (threadIdx.x == 0) {
    mbar_init(&bar.q_full, 1);
    mbar_init(&bar.q_empty, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bar.full[s], 1);
      mbar_init(&bar.empty[s], 1);
    }
    for (int t = 0; t < kTiles; ++t) {
      mbar_init(&bar.s_full[t], 1);
      mbar_init(&bar.p_full[t], 4);
      mbar_init(&bar.o_done[t], 1);
      mbar_init(&bar.o_free[t], 4);
    }
    for (int u = 0; u < 2; ++u) {
      mbar_init(&bar.unit_full[u], 1);
      mbar_init(&bar.unit_empty[u], kUnitReaders);
    }
    mbar_init(&bar.drain, 1);
    mbar_init(&bar.never, 1);
    bar.abort = 0;
    bar.q_loads = 0;
    for (int s = 0; s < kStages; ++s) bar.issued[s] = -1;
    fence_barrier_init();
  }
  if (warp == kWarpTma && lane == 0) {
    prefetch_tensormap(&tmap_q);
    prefetch_tensormap(&tmap_k);
    if (p.k_new != nullptr) prefetch_tensormap(&tmap_kn);
  }
  if (warp == kWarpTmaV && lane == 0) {
    prefetch_tensormap(&tmap_v);
    if (p.k_new != nullptr) prefetch_tensormap(&tmap_vn);
  }
  if (warp == kWarpMma) tmem_alloc(&bar.tmem_base, kTmemCols);
  // q and the metadata were written before the step's first kernel. When that
  // kernel is one of libcb's (which start their dependents only after their own
  // wait on the previous grid), they are visible already and only the cache
  // reads (the TMA warps) wait for a scatter launch; otherwise every thread waits.
  if (!p.metadata_ready && !p.concurrent) grid_dependency_wait();
  tcgen05_fence_before();
  __syncthreads();
  tcgen05_fence_after();
  allow_dependent_launch();
  const uint32_t tmem = bar.tmem_base;
  bool ok = true;

  // ---- teardown, run by every warp at the end of its role (each role ends in its own
  // copy, so that the roles' code shares no join point: their register budgets differ)
  auto teardown = [&]() {
    tcgen05_fence_before();
    __syncthreads();
    if (warp == kWarpMma) {
      tcgen05_fence_after();
      tmem_dealloc(tmem, kTmemCols);
    }
    // If a wait gave up, copies may be in flight that no MMA consumed. The ring's slots
    // are filled in index order and a slot is refilled only after its previous copy was
    // consumed, so only the latest copy of each slot can be in flight: waiting for its
    // phase drains the ring before the CTA's shared memory is released (and likewise the
    // latest query tiles' copy).
    if (threadIdx.x == 0 && *reinterpret_cast<volatile int*>(&bar.abort)) {
      if (bar.q_loads > 0) mbar_wait(&bar.q_full, (uint32_t)((bar.q_loads - 1) & 1));
      for (int s2 = 0; s2 < kStages; ++s2) {
        const int i = bar.issued[s2];
        if (i >= 0) mbar_wait(&bar.full[s2], (uint32_t)((i / kStages) & 1));
      }
    }
    // The last CTA to finish sets the claim counters and the exit counter back to zero for
    // the next step; launched beside the decode kernel, it also waits for the decode grid,
    // so that this grid completes only after it (the combine launch that follows waits for
    // this grid and reads the decode partials).
    if (threadIdx.x == 0 && !p.device_work) {
      if (atomicAdd(p.exit_counter, 1) == (int)gridDim.x - 1) {
        atomicExch(p.exit_counter, 0);
        atomicExch(p.unit_counter, 0);
        atomicExch(p.scatter_counter, 0);
        if (p.concurrent) grid_dependency_wait();
      }
    }
  };

  // Every role reads the CTA's units in the same order from a two-slot ring that the K
  // TMA warp fills: with the work found on the device, the CTA's one unit; otherwise the
  // next unit of the step's list (heaviest first) claimed through an atomic counter, so
  // that a CTA takes a new unit as soon as it can (and CTAs that start late, on SMs a
  // decode grid held, take what is left).
  auto read_unit = [&](int u, UnitDesc& d) -> bool {
    if (!mbar_wait_warp_or_abort(&bar.unit_full[u & 1], (uint32_t)((u >> 1) & 1), &bar.abort))
      return false;
    d = bar.unit[u & 1];
    __syncwarp();
    if (lane == 0) mbar_arrive(&bar.unit_empty[u & 1]);
    return true;
  };

  if (warp >= kWarpTma) {
  // The issuing warpgroup caps its registers (each role branch below ends in its own
  // teardown, so no code after this point is shared with the softmax warps).
  setmaxnreg_dec<kRegsIssue>();
  if (warp == kWarpTma || warp == kWarpTmaV) {
    // =================================================== TMA warps
    // One warp loads the K tiles (ring indices 2j), the other the V tiles (2j + 1):
    // a 16-key page makes 16 boxes per tile, and one warp issuing them all would
    // fall behind the tensor pipe. The K warp also schedules the units and loads their
    // query tiles.
    const int is_v = warp == kWarpTmaV;
    const CUtensorMap* map = is_v ? &tmap_v : &tmap_k;
    const CUtensorMap* nmap = is_v ? &tmap_vn : &tmap_kn;
    const uint4* new_rows = static_cast<const uint4*>(is_v ? p.v_new : p.k_new);
    const uint4* cache = static_cast<const uint4*>(is_v ? p.a.v_cache : p.a.k_cache);
    const bool fuse = p.k_new != nullptr;
    const int BS = p.a.block_size;
    const int box = p.box_keys;
    const int lg_box = __ffs(box) - 1;  // box and block_size are powers of two
    const int lg_bs = __ffs(BS) - 1;
    const int bs_mask = BS - 1;
    const int ppt = kKeys / box;  // pages per key tile
    const int nbox = ppt * kHalves;
    if (p.metadata_ready && !p.concurrent) grid_dependency_wait();  // the step's scatter launch
    int i_base = 0;  // ring index of this unit's K_0
    for (int u = 0; ok; ++u) {
      UnitDesc d;
      if (!is_v) {
        // ---- scheduler (the ring slot is free once every reader is done with unit u - 2)
        if (u >= 2 && !mbar_wait_warp_or_abort(&bar.unit_empty[u & 1], (uint32_t)(((u >> 1) - 1) & 1),
                                               &bar.abort)) {
          ok = false;
          break;
        }
        if (p.device_work) {
          d = u == 0 ? s_first : UnitDesc{-1, 0, 0, 0, 0, 0, 0};
        } else {
          // claimed once the previous unit's loads are all issued (the ring's depth
          // ahead of its products), so that a unit goes to the first CTA that can
          // start it: claimed earlier, a light unit could wait behind a heavy one
          int idx = 0;
          if (lane == 0) idx = atomicAdd(p.unit_counter, 1);
          idx = __shfl_sync(0xffffffffu, idx, 0);
          d = UnitDesc{-1, 0, 0, 0, 0, 0, 0};
          if (idx < p.total_units) {
            const Work w = work_of(p, idx);
            if (w.e >= 0) {
              const PrefillEntry& en = p.entries[w.e];
              d = UnitDesc{en.r, en.q_start, en.q_len, en.seq_len, w.g, w.pair, 1};
            }
          }
        }
        if (lane == 0) {
          bar.unit[u & 1] = d;
          mbar_arrive(&bar.unit_full[u & 1]);
        }
        __syncwarp();
      } else if (!read_unit(u, d)) {
        ok = false;
        break;
      }
      if (!d.live) break;
      const Geo e = geo_of(d, TQ, W);
      const int g = e.g, q_start = e.q_start, seq = e.seq, ctx = e.ctx, kt0 = e.kt0, nkt = e.nkt;
      const int npages_req = (seq + BS - 1) / BS;
      const int32_t* bt = p.a.block_table + (long long)e.r * p.a.bt_stride;
      // page ids of key tile j (lane i < ppt: page i of the tile); checked where
      // they are used, so that the load of the next tile's ids does not stall
      auto tile_pages = [&](int j) -> int {
        const int lp = (((kt0 + j) * kKeys) >> lg_bs) + lane;
        return (lane < ppt && lp < npages_req) ? __ldg(bt + bt_entry(lp, p.a.ring_blocks)) : 0;
      };
      // slot_mapping entries of tile j's keys lane + 32 q that are this step's new
      // positions (ctx <= pos < seq); -1 elsewhere
      auto tile_slots = [&](int j, long long (&sl)[4]) {
        const int key_base = (kt0 + j) * kKeys;
        if (!(fuse && key_base + kKeys > ctx && key_base < seq)) return;  // no new position
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const int pos = key_base + lane + 32 * q4;
          sl[q4] = (pos >= ctx && pos < seq) ? __ldg(p.slot_mapping + q_start + (pos - ctx)) : -1;
        }
      };
      int ids_cur = tile_pages(0);
      long long sl_cur[4], sl_next[4];
      tile_slots(0, sl_cur);
      if (!is_v) {
        // the two query tiles: box (64 of D, the G heads of KV head g, TQ tokens) per tile
        // and half of D lands as the tile's 128 rows (token-major, head-minor) in the
        // 128B-swizzled K-major layout the products read; tokens past the request are
        // never output rows (past T they read as zeros). The buffer is free once the
        // previous unit's last S product is complete.
        if (u >= 1 && !mbar_wait_warp_or_abort(&bar.q_empty, (uint32_t)((u - 1) & 1), &bar.abort)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          mbar_arrive_expect_tx(&bar.q_full, (uint32_t)((e.has_b ? 2 : 1) * kTile));
          for (int t = 0; t < (e.has_b ? 2 : 1); ++t)
            for (int h = 0; h < kHalves; ++h)
              tma_load_3d(sQ + t * kTile + h * kHalfBytes, &tmap_q, &bar.q_full, h * 64, g * G,
                          q_start + (e.qt0 + t) * TQ);
          bar.q_loads = u + 1;  // read by the drain after the CTA's final barrier
        }
        __syncwarp();
      }
      for (int j = 0; j < nkt; ++j) {
        const int i = i_base + 2 * j + is_v;
        const int s = i % kStages;
        uint8_t* dst = sRing + s * kTile;
        const int key_base = (kt0 + j) * kKeys;
        // the next tile's page ids and slots are read while this one waits for its slot
        const int ids_next = j + 1 < nkt ? tile_pages(j + 1) : 0;
        if (j + 1 < nkt) tile_slots(j + 1, sl_next);
        if (i >= kStages &&
            !mbar_wait_warp_or_abort(&bar.empty[s], (uint32_t)(((i / kStages) - 1) & 1), &bar.abort)) {
          ok = false;
          break;
        }
        // ---- where each page box of the tile comes from. A new position (ctx <= pos <
        // seq) whose slot is its own holds k_new's row after this step, so it is read from
        // k_new; any other position from the cache (not written in this step). Tiles of
        // context only (the common case) skip the test: this warp's issue rate bounds the
        // ring's refill rate.
        const bool tile_new = fuse && key_base + kKeys > ctx && key_base < seq;  // warp-uniform
        unsigned bad[4] = {0u, 0u, 0u, 0u};  // bit kk: key key_base + kk is new, slot not its own
        int src = 0;  // lane i < ppt: page i from 0: the cache (or zeros past the request),
                      // 1: a box of k_new rows, 2: row by row (straddles ctx or foreign slot)
        unsigned gen = 0u;
        if (tile_new) {
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            const int kk = lane + 32 * q4;
            const int pos = key_base + kk;
            const int pgk = __shfl_sync(0xffffffffu, ids_cur, (kk >> lg_box) & 31);
            const bool isnew = pos >= ctx && pos < seq;
            bad[q4] = __ballot_sync(0xffffffffu,
                                    isnew && sl_cur[q4] != (long long)pgk * BS + (pos & bs_mask));
          }
          const int kp = key_base + (lane << lg_box);
          if (lane < ppt && kp < seq && kp + box > ctx) {
            bool pbad = false;
#pragma unroll
            for (int w4 = 0; w4 < 4; ++w4) {
              const int lo = max(lane << lg_box, 32 * w4), hi = min((lane << lg_box) + box, 32 * w4 + 32);
              if (lo < hi) {
                const unsigned bits = bad[w4] >> (lo - 32 * w4);
                pbad |= (hi - lo == 32 ? bits : (bits & ((1u << (hi - lo)) - 1u))) != 0u;
              }
            }
            src = (kp >= ctx && !pbad) ? 1 : 2;
          }
          gen = __ballot_sync(0xffffffffu, src == 2);
        }
        if (gen != 0u) {
          copy_rows<D>(dst, gen, ids_cur, bad[0], bad[1], bad[2], bad[3], key_base, ctx, seq, q_start, g,
                       Hkv, BS, box, new_rows, cache, p.a.num_blocks, p.a.error_word);
          // the tensor cores read these rows through the async proxy
          fence_proxy_async_smem();
          __syncwarp();
        }
        if (lane == 0) {
          const int tma_bytes = kTile - __popc(gen) * kHalves * box * 128;
          mbar_arrive_expect_tx(&bar.full[s], (uint32_t)tma_bytes);
          bar.issued[s] = (int)i;  // read by the drain after the CTA's final barrier
        }
        __syncwarp();  // the expect_tx is registered first
        {
          // lane b < nbox loads box b (page b / kHalves, half b % kHalves of head_dim); a
          // page past the request, or past the pool, reads as zeros
          const int key0 = BS > kKeys ? (key_base & bs_mask) : 0;
          const int page = lane / kHalves;
          const int half = lane % kHalves;
          int pgb = __shfl_sync(0xffffffffu, ids_cur, page & 31);
          const int srcb = tile_new ? __shfl_sync(0xffffffffu, src, page & 31) : 0;
          if (lane < nbox && srcb != 2) {
            uint8_t* bdst = dst + half * kHalfBytes + page * box * 128;
            if (srcb == 1) {
              tma_load_3d(bdst, nmap, &bar.full[s], half * 64, g, q_start + (key_base + (page << lg_box) - ctx));
            } else {
              if ((((kt0 + j) * kKeys) >> lg_bs) + page >= npages_req) {
                pgb = p.a.num_blocks;
              } else if (pgb < 0 || pgb >= p.a.num_blocks) {
                record_error(p.a.error_word, 0x1);
                pgb = p.a.num_blocks;
              }
              tma_load_4d(bdst, map, &bar.full[s], half * 64, key0, g, pgb);
            }
          }
        }
        __syncwarp();
        ids_cur = ids_next;
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) sl_cur[q4] = sl_next[q4];
      }
      if (!ok) break;
      i_base += 2 * nkt;
    }
    if (!ok && lane == 0) {
      record_error(p.a.error_word, 0x4);
      set_abort(&bar.abort);
    }
    teardown();
  } else if (warp == kWarpMma) {
    // =================================================== MMA issuer
    // The whole warp runs this loop (the descriptors stay warp-uniform); one
    // elected lane issues the MMAs and the commits that track them.
    constexpr uint32_t idS = umma_idesc_bf16(kRows, kKeys, false);
    constexpr uint32_t idO = umma_idesc_bf16(kRows, D, true);
    // descriptors: K-major Q and K tiles, N-major V tiles (the start address >> 4
    // sits in the low bits, so moving within shared memory is an addition)
    const uint64_t dQ = umma_desc_sw128_base(16, 1024) | (smem_u32(sQ) >> 4);
    const uint64_t dK = umma_desc_sw128_base(16, 1024) | (smem_u32(sRing) >> 4);
    const uint64_t dV = umma_desc_sw128_base(kHalfBytes, 1024) | (smem_u32(sRing) >> 4);
    auto slot_ready = [&](int i) {
      return mbar_wait_warp_or_abort(&bar.full[i % kStages], (uint32_t)((i / kStages) & 1),
                                     &bar.abort);
    };
    // S_t = Q_t K^T with K in ring slot i; its completion is signalled on s_full[t]
    auto qk = [&](int t, int i) {
      const uint64_t dq = dQ + (uint64_t)(t * (kTile >> 4));
      const uint64_t dk = dK + (uint64_t)((i % kStages) * (kTile >> 4));
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        const uint32_t off = ((ks >> 2) * kHalfBytes + (ks & 3) * 32) >> 4;
        umma_bf16_elect(tmem + t * kKeys, dq + off, dk + off, idS, ks > 0 ? 1u : 0u);
      }
      umma_commit_elect(&bar.s_full[t]);
    };
    // O_t += P_t V with P in the first 64 columns of S_t and V in ring slot i
    auto pv = [&](int t, int i, bool acc) {
      const uint64_t dv = dV + (uint64_t)((i % kStages) * (kTile >> 4));
#pragma unroll
      for (int ks = 0; ks < kKeys / 16; ++ks)
        umma_bf16_tmem_a_elect(tmem + 2 * kKeys + t * D, tmem + t * kKeys + ks * 8,
                               dv + (uint64_t)(ks * (2048 >> 4)), idO, (acc || ks > 0) ? 1u : 0u);
    };
    int i_base = 0;
    int pwaits[kTiles] = {0, 0};  // p_full waits done so far (phase parity)
    int olive[kTiles] = {0, 0};   // units so far in which query tile t had rows
    for (int u = 0; ok; ++u) {
      UnitDesc d;
      if (!read_unit(u, d)) {
        ok = false;
        break;
      }
      if (!d.live) break;
      const Geo e = geo_of(d, TQ, W);
      const int nkt = e.nkt;
      const bool has_b = e.has_b;
      ok = mbar_wait_warp_or_abort(&bar.q_full, (uint32_t)(u & 1), &bar.abort) && slot_ready(i_base);
      if (!ok) break;
      tcgen05_fence_after();
      qk(0, i_base);
      if (has_b) qk(1, i_base);
      umma_commit_elect(&bar.empty[i_base % kStages]);
      if (nkt == 1) umma_commit_elect(&bar.q_empty);  // the unit's last S products
      for (int j = 0; j < nkt && ok; ++j) {
        const int iv = i_base + 2 * j + 1;  // V_j
        const int ik = i_base + 2 * j + 2;  // K_{j+1}
        const bool more = j + 1 < nkt;
        // the loads are waited for before P, the one wait that depends on the softmax;
        // before the unit's first PV_t the epilogue of O_t's previous unit must be done
        if (!slot_ready(iv) || (more && !slot_ready(ik)) ||
            !mbar_wait_warp_or_abort(&bar.p_full[0], (uint32_t)(pwaits[0]++ & 1), &bar.abort) ||
            (j == 0 && olive[0] > 0 &&
             !mbar_wait_warp_or_abort(&bar.o_free[0], (uint32_t)((olive[0] - 1) & 1), &bar.abort))) {
          ok = false;
          break;
        }
        tcgen05_fence_after();
        pv(0, iv, j > 0);
        if (!more) umma_commit_elect(&bar.o_done[0]);
        if (!has_b) umma_commit_elect(&bar.empty[iv % kStages]);
        if (more) qk(0, ik);
        if (more && !has_b && j + 2 == nkt) umma_commit_elect(&bar.q_empty);
        if (has_b) {
          if (!mbar_wait_warp_or_abort(&bar.p_full[1], (uint32_t)(pwaits[1]++ & 1), &bar.abort) ||
              (j == 0 && olive[1] > 0 &&
               !mbar_wait_warp_or_abort(&bar.o_free[1], (uint32_t)((olive[1] - 1) & 1), &bar.abort))) {
            ok = false;
            break;
          }
          tcgen05_fence_after();
          pv(1, iv, j > 0);
          if (!more) umma_commit_elect(&bar.o_done[1]);
          umma_commit_elect(&bar.empty[iv % kStages]);
          if (more) qk(1, ik);
          if (more && j + 2 == nkt) umma_commit_elect(&bar.q_empty);
        }
        if (more) umma_commit_elect(&bar.empty[ik % kStages]);
      }
      if (!ok) break;
      ++olive[0];
      if (has_b) ++olive[1];
      i_base += 2 * nkt;
    }
    if (!ok && lane == 0) {
      record_error(p.a.error_word, 0x4);
      set_abort(&bar.abort);
    }
    // every MMA this warp issued has completed before the TMEM is released (the
    // commit tracks them all; it completes whether or not the loop ran to its end)
    umma_commit_elect(&bar.drain);
    mbar_wait_warp(&bar.drain, 0);
    teardown();
  } else {
    teardown();  // warp 11
  }
  } else {
    setmaxnreg_inc<kRegsSoftmax>();
    // =================================================== softmax warpgroups
    const int t = warp >> 2;             // query tile of this group
    const int row = threadIdx.x & (kRows - 1);  // TMEM lane = tile row
    const uint32_t lane_addr = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_addr + t * kKeys;
    const uint32_t tO = tmem + lane_addr + 2 * kKeys + t * D;
    int i_base = 0;
    int swaits = 0;  // s_full[t] waits so far (phase parity)
    const bool copy_rows_after = p.k_new != nullptr && !p.device_work;  // the row copy below
    bool claimed = false;  // its first part is claimed already (lane 0: first_part)
    int first_part = 0;
    int owaits = 0;  // o_done[t] waits so far
    for (int u = 0; ok; ++u) {
      // The unit stays in its ring slot until this group is done with it (the slot is
      // released at the unit's end), so that its fields are read from shared memory where
      // they are used instead of being held in registers across the key loop.
      if (!mbar_wait_warp_or_abort(&bar.unit_full[u & 1], (uint32_t)((u >> 1) & 1), &bar.abort)) {
        ok = false;
        break;
      }
      const volatile UnitDesc* ud = &bar.unit[u & 1];
#define CB_UNIT_GEO() geo_of(ud->r, ud->q_start, ud->q_len, ud->seq_len, ud->g, ud->pair, TQ, W)
#define CB_RELEASE_UNIT()                                 \
  do {                                                    \
    __syncwarp();                                         \
    if (lane == 0) mbar_arrive(&bar.unit_empty[u & 1]);   \
  } while (0)
      if (!ud->live) {
        CB_RELEASE_UNIT();
        break;
      }
      int kt0, nkt, seq, min_kv, max_kv, tile_max_kv_min, tile_min_kv_max;
      {
        const Geo e = CB_UNIT_GEO();
        const int unit_nkt = e.nkt;
        const bool tile_live = t == 0 || e.has_b;
        if (!tile_live) {  // this unit has no tile B
          i_base += 2 * unit_nkt;
          CB_RELEASE_UNIT();
          continue;
        }
        kt0 = e.kt0;
        nkt = e.nkt;
        seq = e.seq;
        const int tok0 = (e.qt0 + t) * TQ;
        const int qpos = e.ctx + tok0 + row / G;
        max_kv = min(qpos, e.seq - 1);
        min_kv = W > 0 ? max(0, qpos - W + 1) : 0;
        // keys every row of the tile attends: [tile_min_kv_max, tile_max_kv_min]
        const int tok_end = min(e.q_len, tok0 + TQ);
        tile_max_kv_min = min(e.ctx + tok0, e.seq - 1);
        tile_min_kv_max = W > 0 ? max(0, e.ctx + tok_end - 1 - W + 1) : 0;
      }
      i_base += 2 * nkt;
      const float sl2 = p.a.scale_log2;
      float m_ref = -FLT_MAX;
      float l = 0.f;
      // test hook: the group's first wait runs out (nothing arrives at bar.never)
      if (u == 0 && p.a.test_expire_wait && !mbar_wait_warp_polls(&bar.never, 0, kTestExpiryPolls))
        ok = false;
      for (int j = 0; j < nkt && ok; ++j) {
        if (!mbar_wait_warp_or_abort(&bar.s_full[t], (uint32_t)(swaits++ & 1), &bar.abort)) {
          ok = false;
          break;
        }
        tcgen05_fence_after();
        uint32_t sr[kKeys];
#pragma unroll
        for (int c0 = 0; c0 < kKeys; c0 += 32)
          tmem_ld32(tS + c0, *reinterpret_cast<uint32_t(*)[32]>(sr + c0));
        tmem_wait_ld();
        float* sv = reinterpret_cast<float*>(sr);
        // mask (bounds only; tiles inside every row's range need none) and row
        // maximum of the raw scores (the scale is positive, so it commutes with max)
        const int key_base = (kt0 + j) * kKeys;
        if (key_base < tile_min_kv_max || key_base + kKeys - 1 > tile_max_kv_min) {
#pragma unroll
          for (int c = 0; c < kKeys; ++c) {
            const int key = key_base + c;
            if (key < min_kv || key > max_kv) sv[c] = -INFINITY;
          }
        }
        float mx8[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) mx8[k] = fmax3(sv[k], sv[8 + 2 * k], sv[9 + 2 * k]);
#pragma unroll
        for (int c = 24; c < kKeys; c += 2) mx8[(c >> 1) & 7] = fmax3(mx8[(c >> 1) & 7], sv[c], sv[c + 1]);
        const float mx = fmax3(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(mx8[3], mx8[4], mx8[5]),
                               fmaxf(mx8[6], mx8[7])) * sl2;
        const bool need = mx > m_ref + kRescaleLog2;
        const float alpha = need ? ex2_approx(m_ref - mx) : 1.f;
        if (need) m_ref = mx;
        // p = 2^(s * scale_log2 - m): one SFU op per score, the exponent arguments and the
        // row sum in packed pairs (the SFU's 4 cycles per warp instruction bound this phase;
        // packing frees issue slots around them: ~10% off the phase)
        float sum8[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) sum8[k] = 0.f;
#pragma unroll
        for (int c = 0; c < kKeys; c += 2) {
          float x0, x1;
          ffma2(x0, x1, sv[c], sv[c + 1], sl2, -m_ref);
          sv[c] = ex2_approx(x0);
          sv[c + 1] = ex2_approx(x1);
          fadd2(sum8[c & 7], sum8[(c & 7) + 1], sv[c], sv[c + 1]);
        }
        const float sum = ((sum8[0] + sum8[1]) + (sum8[2] + sum8[3])) +
                          ((sum8[4] + sum8[5]) + (sum8[6] + sum8[7]));
        l = l * alpha + sum;
        // P row as bf16 pairs over the first 64 columns of S_t (lane = row)
#pragma unroll
        for (int c0 = 0; c0 < kKeys; c0 += 32) {
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) pk[i] = pack_bf16x2(sv[c0 + 2 * i], sv[c0 + 2 * i + 1]);
          tmem_st16(tS + c0 / 2, pk);
        }
        // O belongs to this group again (S_t of this tile was issued after the
        // previous PV_t): rescale it when a row's maximum was raised, before the
        // next PV_t is issued (done after the P store, when the scores are dead)
        if (j > 0 && __any_sync(0xffffffffu, need)) {
#pragma unroll
          for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t o32[32];
            tmem_ld32(tO + c0, o32);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) o32[i] = __float_as_uint(__uint_as_float(o32[i]) * alpha);
            tmem_st32(tO + c0, o32);
          }
        }
        // V rows past the end of the sequence hold unrelated data: zero them so
        // that 0 * V cannot produce a NaN (row index = key index in the tile).
        // Each group does it before its own P is signalled (the other group may
        // write the same zeros at the same time), so before either PV reads V.
        if (key_base + kKeys > seq) {
          const int iv = i_base - 2 * (nkt - j) + 1;  // V_j of this unit
          if (!mbar_wait_warp_or_abort(&bar.full[iv % kStages], (uint32_t)((iv / kStages) & 1),
                                       &bar.abort)) {
            ok = false;
            break;
          }
          if (key_base + row >= seq) {
#pragma unroll
            for (int h = 0; h < kHalves; ++h)
#pragma unroll
              for (int c = 0; c < 8; ++c)
                *reinterpret_cast<uint4*>(sRing + (iv % kStages) * kTile + h * kHalfBytes + row * 128 +
                                          c * 16) = make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
        }
        tmem_wait_st();
        tcgen05_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar.p_full[t]);
      }
      // ---- epilogue: O / l for the rows of this tile. The rows' output offsets are
      // computed while the last PV product runs (~600 cycles after the wait otherwise).
      const int q4 = lane & 3;
      long long orow[4];  // bf16 offset of rows 4a .. 4a + 3 of the warp, -1 past q_len
      {
        const Geo e = CB_UNIT_GEO();
        const int lg = __ffs(G) - 1;
#pragma unroll
        for (int s4 = 0; s4 < 4; ++s4) {
          const int r = (warp & 3) * 32 + 4 * (lane >> 2) + s4;  // tile row
          const int tok = (e.qt0 + t) * TQ + (r >> lg);
          orow[s4] = tok < e.q_len ? ((long long)(e.q_start + tok) * p.a.num_q_heads + e.g * G +
                                      (r & (G - 1))) * D + q4 * 16
                                   : -1;
        }
      }
      // When the next unit is already published as the end of the list, the first part of
      // the row copy that follows is claimed now: the claim's round trip to L2 overlaps
      // the epilogue instead of following it on the CTA's last unit.
      if (copy_rows_after && !claimed) {
        int last = 0;
        if (lane == 0 && mbar_try_wait(&bar.unit_full[(u + 1) & 1], (uint32_t)(((u + 1) >> 1) & 1)) &&
            !bar.unit[(u + 1) & 1].live) {
          last = 1;
          first_part = atomicAdd(p.scatter_counter, 1);
        }
        claimed = __shfl_sync(0xffffffffu, last, 0) != 0;
      }
      if (ok && !mbar_wait_warp_or_abort(&bar.o_done[t], (uint32_t)(owaits++ & 1), &bar.abort))
        ok = false;
      if (ok) {
        tcgen05_fence_after();
        const float inv = l > 0.f ? 1.f / l : 0.f;
        // O / l as bf16 in whole 128-byte lines. Each lane holds its own row (TMEM lane =
        // row); a transpose of 32-byte pieces within each group of four lanes gives lane
        // 4a + q piece q of rows 4a .. 4a + 3 of the warp, so that one store instruction
        // writes 8 rows x 128 contiguous bytes instead of 32 rows x 16 bytes (the stores of
        // one row per lane kept the LSU busy ~4000 cycles per unit).
        const bool wide = (reinterpret_cast<uintptr_t>(p.a.out) & 31) == 0;
        __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.a.out);
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 64) {
          uint32_t o0[32], o1[32];
          tmem_ld32(tO + c0, o0);
          tmem_ld32(tO + c0 + 32, o1);
          tmem_wait_ld();
          uint32_t w[32];  // piece k = words 8k .. 8k + 7 = columns c0 + 16k .. c0 + 16k + 15
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            w[i] = pack_bf16x2(__uint_as_float(o0[2 * i]) * inv, __uint_as_float(o0[2 * i + 1]) * inv);
            w[16 + i] = pack_bf16x2(__uint_as_float(o1[2 * i]) * inv, __uint_as_float(o1[2 * i + 1]) * inv);
          }
          // in-quad transpose: at lane distance d, the lane whose bit d is set swaps its
          // pieces with bit d clear for its partner's pieces with bit d set
#pragma unroll
          for (int d = 2; d >= 1; d >>= 1) {
            const bool hi = (lane & d) != 0;
#pragma unroll
            for (int k0 = 0; k0 < 4; ++k0) {
              if (k0 & d) continue;
              const int k1 = k0 | d;
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const uint32_t x = hi ? w[8 * k0 + i] : w[8 * k1 + i];
                const uint32_t y = __shfl_xor_sync(0xffffffffu, x, d);
                if (hi) w[8 * k0 + i] = y;
                else w[8 * k1 + i] = y;
              }
            }
          }
          // now piece s4 of this lane = columns c0 + 16 q .. + 15 of row 4a + s4
#pragma unroll
          for (int s4 = 0; s4 < 4; ++s4) {
            if (orow[s4] < 0) continue;
            __nv_bfloat16* dst = out + orow[s4] + c0;
            if (wide) {
              st_global_v8(dst, w[8 * s4 + 0], w[8 * s4 + 1], w[8 * s4 + 2], w[8 * s4 + 3],
                           w[8 * s4 + 4], w[8 * s4 + 5], w[8 * s4 + 6], w[8 * s4 + 7]);
            } else {
              *reinterpret_cast<uint4*>(dst) = make_uint4(w[8 * s4 + 0], w[8 * s4 + 1], w[8 * s4 + 2], w[8 * s4 + 3]);
              *reinterpret_cast<uint4*>(dst + 8) = make_uint4(w[8 * s4 + 4], w[8 * s4 + 5], w[8 * s4 + 6], w[8 * s4 + 7]);
            }
          }
        }
        // O_t is read: the next unit's products may overwrite it
        tcgen05_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar.o_free[t]);
      } else if (lane == 0) {
        record_error(p.a.error_word, 0x4);
        set_abort(&bar.abort);
      }
      if (!ok) break;
      CB_RELEASE_UNIT();
    }
#undef CB_UNIT_GEO
#undef CB_RELEASE_UNIT
    if (!ok && lane == 0) {
      record_error(p.a.error_word, 0x4);
      set_abort(&bar.abort);
    }
    // ---- the step's new K and V rows to their slots (a slot below zero is skipped, one
    // past the pool recorded and skipped). Nothing in the step reads these positions from
    // the cache (the TMA warps read them from k_new), so the copy may run at any time: the
    // softmax warps of CTAs with no attention work left claim it a quarter of a unit's
    // tokens for its KV head at a time, so that it runs while the longest units compute
    // and competes with no product of its own CTA. The parts of all units cover every
    // (token, KV head) of the listed requests once.
    if (ok && copy_rows_after) {
      constexpr int kParts = 4;
      constexpr int kRowChunks = D / 8;  // 16-byte chunks of one head's row
      constexpr int kPerTok = 2 * kRowChunks;
      static_assert(32 % kPerTok == 0 || kPerTok == 32, "a lane keeps one chunk of the row");
      constexpr int kTokPass = 32 / kPerTok;  // tokens per pass of the warp
      constexpr int kBatch = 8;
      const long long num_slots = (long long)p.a.num_blocks * p.a.block_size;
      const int rem = lane % kPerTok;  // the same 16-byte chunk of every token it copies
      const int sub = lane / kPerTok;
      const int per = kTiles * TQ / kParts;  // TQ = 128 / G tokens, so 4 or more per part
      const int n_parts = p.total_units * kParts;
      for (;;) {
        int it = 0;
        if (lane == 0) it = claimed ? first_part : atomicAdd(p.scatter_counter, 1);
        claimed = false;
        it = __shfl_sync(0xffffffffu, it, 0);
        if (it >= n_parts) break;
        const Work w = work_of(p, it / kParts);
        if (w.e < 0) continue;
        const PrefillEntry& en = p.entries[w.e];
        const int a0 = kTiles * w.pair * TQ + (it % kParts) * per;
        const int ntok = min(en.q_len - a0, per);
        const uint4* src = static_cast<const uint4*>(rem < kRowChunks ? p.k_new : p.v_new) +
                           (long long)w.g * kRowChunks + rem % kRowChunks;
        uint4* dst = static_cast<uint4*>(rem < kRowChunks ? p.a.k_cache : p.a.v_cache) +
                     (long long)w.g * kRowChunks + rem % kRowChunks;
        const long long tk_first = (long long)en.q_start + a0;
        for (int k0 = sub; k0 < ntok; k0 += kTokPass * kBatch) {
          uint4 v[kBatch];
          long long sl[kBatch];
#pragma unroll
          for (int b = 0; b < kBatch; ++b) {
            const int k = k0 + kTokPass * b;
            sl[b] = -1;
            if (k < ntok) {
              sl[b] = __ldg(p.slot_mapping + tk_first + k);
              v[b] = __ldg(src + (tk_first + k) * (Hkv * kRowChunks));
            }
          }
#pragma unroll
          for (int b = 0; b < kBatch; ++b) {
            if (sl[b] >= 0) {
              if (sl[b] < num_slots)
                dst[sl[b] * (Hkv * kRowChunks)] = v[b];
              else if (rem == 0)
                record_error(p.a.error_word, 0x2);
            }
          }
        }
      }
    }
    teardown();
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
  // the step's new rows [T, Hkv, D] as (d, head, token); box: 64 of d, one head,
  // box_keys tokens -- the same shared-memory rows as a page box of the cache
  CUtensorMap mkn = mk, mvn = mv;  // unused without new rows
  if (p.k_new != nullptr) {
    cuuint64_t nd[3] = {(cuuint64_t)D, (cuuint64_t)a.num_kv_heads, (cuuint64_t)a.num_tokens};
    cuuint64_t ns[2] = {(cuuint64_t)D * e, (cuuint64_t)a.num_kv_heads * D * e};
    cuuint32_t nb[3] = {64, 1, (cuuint32_t)p.box_keys};
    err = encode(&mkn, const_cast<void*>(p.k_new), 3, nd, ns, nb);
    if (err == cudaSuccess) err = encode(&mvn, const_cast<void*>(p.v_new), 3, nd, ns, nb);
    if (err != cudaSuccess) return err;
  }
  // q [T, Hq, D] as (d, head, token); box: 64 of d, the G heads of a KV head, the
  // tokens of a 128-row tile
  CUtensorMap mq;
  {
    const int G = a.num_q_heads / a.num_kv_heads;
    if (G < 1 || kRows % G != 0 || p.tile_tokens != kRows / G) return cudaErrorInvalidValue;
    cuuint64_t qd[3] = {(cuuint64_t)D, (cuuint64_t)a.num_q_heads, (cuuint64_t)a.num_tokens};
    cuuint64_t qs[2] = {(cuuint64_t)D * e, (cuuint64_t)a.num_q_heads * D * e};
    cuuint32_t qb[3] = {64, (cuuint32_t)G, (cuuint32_t)p.tile_tokens};
    err = encode(&mq, const_cast<void*>(a.q), 3, qd, qs, qb);
    if (err != cudaSuccess) return err;
  }
  auto kern = prefill_tile_kernel<D>;
  static bool attr_set = false;
  constexpr size_t smem = smem_bytes<D>();
  if (!attr_set) {
    // the register split inside the kernel assumes kRegsLaunch registers per thread at
    // launch; with fewer, the softmax warps' increase would wait for registers forever
    cudaFuncAttributes fa;
    err = cudaFuncGetAttributes(&fa, kern);
    if (err != cudaSuccess) return err;
    if (fa.numRegs != kRegsLaunch) return cudaErrorInvalidConfiguration;
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    attr_set = true;
  }
  return launch_pdl(kPrefillTc, kern, dim3(p.grid), dim3(kThreads), smem, s, mk, mv, mkn, mvn,
                    mq, p);
}

}  // namespace

size_t prefill_smem_bytes(int head_dim) {
  return head_dim == 64 ? smem_bytes<64>() : smem_bytes<128>();
}

int prefill_ctas(int n_qtiles, int num_kv_heads) {
  return ((n_qtiles + kTiles - 1) / kTiles) * num_kv_heads;
}

int prefill_ctas_bound(int num_tokens, int num_requests, int tile_tokens, int num_kv_heads) {
  // over the n <= min(R, T / 2) requests with q_len > 1:
  // sum of ceil(ceil(q_len / TQ) / 2) <= (sum q_len / TQ + 2 n) / 2
  const long long n = num_requests < num_tokens / 2 ? num_requests : num_tokens / 2;
  const long long tiles = (long long)num_tokens / tile_tokens + 2 * n;
  return (int)((tiles + 1) / 2) * num_kv_heads;
}

cudaError_t prepare_prefill(int head_dim) {
  if (head_dim == 64)
    return cudaFuncSetAttribute(prefill_tile_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)smem_bytes<64>());
  return cudaFuncSetAttribute(prefill_tile_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)smem_bytes<128>());
}

cudaError_t launch_prefill(const PrefillArgs& p, cudaStream_t stream) {
  if (p.grid <= 0) return cudaSuccess;
  if (p.a.head_dim == 64) return launch_d<64>(p, stream);
  return launch_d<128>(p, stream);
}

}  // namespace cb
