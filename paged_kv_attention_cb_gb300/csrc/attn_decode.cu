// Decode rows (q_len == 1) of the step: split-KV paged attention, bf16.
//
// What it computes is the decode case of the per-block pseudocode of
// "Continuous Batching" (languisher.top), section "Extension: the vLLM v1
// implementation": context_len = seq_len - 1, the single query attends
// kv_pos 0 .. context_len (or the last sliding_window positions), each
// resolved through block_table[req][kv_pos / BLOCK_SIZE] at offset
// kv_pos % BLOCK_SIZE. Decode is memory-bound ("Continuous batching
// mechanics", d9bl.com, section "A single request on a GPU"), so the design
// goal is to stream every attended K/V byte from HBM exactly once at full
// bandwidth:
//
// * Work partition. The decode requests' key blocks (16 keys of one request,
//   all KV heads) are numbered in request order, u = 0 .. U-1, and CTA b of C
//   takes the contiguous range [b*U/C, (b+1)*U/C): every CTA streams the same
//   number of bytes whatever the length mix, and a long request is split
//   across CTAs (split-KV). The host places each CTA's start (or, for a
//   captured graph, each CTA finds it with a block scan over the decode
//   lengths); the CTA then walks forward. A piece of a request inside one CTA
//   is a segment; a request that lies in one CTA writes its output directly,
//   otherwise each segment writes an unnormalised partial (m, l, o), and the
//   combine kernel that follows on the stream merges them (log-sum-exp), one
//   CTA per (split request, KV head), so a long request's merge is spread
//   over several SMs instead of falling on the one that finishes last.
// * GQA packing. One CTA covers up to 8 KV heads (one consumer warp each) and
//   all G query heads of each KV head, so K/V are read once for the group.
// * Staging. A producer warp moves each 16-key block of all the CTA's heads
//   with four 128B-swizzled TMA tile loads (K and V, two 64-element halves of
//   D) into a STAGES-deep ring of shared-memory buffers guarded by mbarriers;
//   the request's query rows arrive by a 1-D bulk copy into a 2-slot ring.
//   With 8-key pages a block is two pages: two loads of 8 keys each, which
//   land as rows (page, head, key) instead of (head, key).
// * Contraction. Per warp and block: S^T (16 keys x 8 heads) = K Q^T and
//   O^T (D x 8 heads) += V^T P^T on mma.sync m16n8k16 (bf16 in, fp32
//   accumulate); the key axis is the M dimension so a group of up to 8 query
//   heads fills the N = 8 columns (G = 16: two such column blocks, sharing each
//   K and V fragment). P^T goes from the accumulator layout to the B-operand
//   layout with movmatrix. Softmax statistics are per column, kept per lane and
//   reduced with warp shuffles.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <float.h>

#include "common.cuh"
#include "decode.h"
#include "launch.h"
#include "sm100_ptx.cuh"

namespace cb {

namespace {

constexpr int kKB = 16;  // keys per block (stage)

struct SegDesc {
  int r;       // request (-1: no more segments)
  int kb0;     // first key block (absolute, within the request)
  int kb1;     // one past the last key block
  int t;       // packed query row of the request
  int lo;      // first attended key (window start)
  int hi;      // last attended key (= seq_len - 1)
  int slot;    // partial slot (r + CTA index)
  int direct;  // 1: the request lies wholly in this CTA
};

struct DecodeSmem {
  uint64_t full[kDecodeMaxStages];
  uint64_t empty[kDecodeMaxStages];
  uint64_t qfull[2];
  uint64_t qempty[2];
  uint64_t never;  // nothing arrives here: the test hook's wait on it runs out
  SegDesc seg[2];
  long long scan[16];
  long long total_u;
  int first_r;
  long long first_u;
  int abort_flag;
};

CB_DEV int kb_lo_of(int seq, int window) {
  const int lo = window > 0 ? max(0, seq - window) : 0;
  return lo / kKB;
}

// Row of (local head hl, key k of the 16-key block) in a staged K or V half: (head, key)
// for pages of 16 keys or more, (page, head, key) for 8-key pages. Rows are 128 bytes
// and the 128B swizzle depends on the row's index modulo 8, which is k mod 8 either way.
CB_DEV int stage_row(bool pages8, int hb, int hl, int k) {
  return pages8 ? ((k >> 3) * hb + hl) * 8 + (k & 7) : hl * kKB + k;
}

// Key blocks a decode query of a request of seq_len `seq` attends.
CB_DEV int units_of(int seq, int window) { return (seq - 1) / kKB - kb_lo_of(seq, window) + 1; }

// Key blocks of request r if it is a decode request, else 0.
// (The three loads are independent: one memory round trip.)
CB_DEV int decode_units(const StepArgs& a, int r, int* seq_out, int* t_out) {
  const int q0 = __ldg(a.query_start_loc + r);
  const int q1 = __ldg(a.query_start_loc + r + 1);
  const int seq = __ldg(a.seq_lens + r);
  *seq_out = seq;
  *t_out = q0;
  if (q1 - q0 != 1 || seq <= 0) return 0;
  return units_of(seq, a.sliding_window);
}

// CTAs a partition of U key blocks uses out of a launch of C: at least
// kDecodeMinBlocksPerCta blocks each, so that a small step is not split into more
// segments than its combine can merge quickly.
CB_DEV int decode_ctas_used(long long U, int C) {
  const long long want = (U + kDecodeMinBlocksPerCta - 1) / kDecodeMinBlocksPerCta;
  return (int)(want < C ? want : C);
}

// CTA that owns global key block u (ranges [b*U/C, (b+1)*U/C)).
CB_DEV int cta_of(long long u, long long U, int C) {
  return (int)(((u + 1) * (long long)C + U - 1) / U) - 1;
}

CB_DEV long long warp_incl_scan(long long v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const long long n = __shfl_up_sync(0xffffffffu, v, off);
    if (lane >= off) v += n;
  }
  return v;
}

}  // namespace

template <int D, int G>
__global__ void __launch_bounds__(kDecodeMaxHeads * 32 + 32, 1)
decode_split_kernel(const __grid_constant__ CUtensorMap tmap_k,
                    const __grid_constant__ CUtensorMap tmap_v, const DecodeArgs p) {
  static_assert(D == 64 || D == 128, "head_dim");
  static_assert(G == 1 || G == 2 || G == 4 || G == 8 || G == 16, "group");
  constexpr int NB = (G + 7) / 8;  // 8-head column blocks
  constexpr int kHalves = D / 64;
  constexpr int kKSteps = D / 16;
  extern __shared__ __align__(1024) uint8_t smem_dyn[];
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
  const int HB = p.heads_per_cta;
  const int box_bytes = HB * kKB * 128;  // one 64-element half of D, all heads, 16 keys
  uint8_t* stages = base;
  uint8_t* qring = base + p.stages * p.stage_bytes;
  DecodeSmem& sm = *reinterpret_cast<DecodeSmem*>(qring + 2 * p.q_slot_bytes);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int nthreads = blockDim.x;
  const int b = blockIdx.x;
  const int hg = blockIdx.y;
  int C = p.num_ctas;
  long long U = p.total_units;
  const int R = p.a.num_requests;

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], HB);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&sm.qfull[s], 1);
      mbar_init(&sm.qempty[s], HB);
    }
    mbar_init(&sm.never, 1);
    sm.first_r = -1;
    sm.first_u = 0;
    sm.abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == HB && lane == 0) {
    prefetch_tensormap(&tmap_k);
    prefetch_tensormap(&tmap_v);
  }
  // The metadata (and q) were written before the step's first kernel: when
  // that kernel is libcb's own scatter, which lets this grid start only after
  // its own wait on the previous grid, they are visible already and only the
  // cache reads (the producer's TMA) must wait for the scatter. Otherwise this
  // is the step's first kernel and every thread waits.
  if (!p.metadata_ready) grid_dependency_wait();
  __syncthreads();
  if (p.units_on_device) {
    // the decode requests' key blocks, summed over the step from the device metadata
    long long part = 0;
    for (int r = threadIdx.x; r < R; r += nthreads) {
      int seq = 0, t = 0;
      part += decode_units(p.a, r, &seq, &t);
    }
    part = warp_incl_scan(part);
    if (lane == 31) sm.scan[warp] = part;
    __syncthreads();
    if (threadIdx.x == 0) {
      long long tot = 0;
      for (int w = 0; w < (nthreads >> 5); ++w) tot += sm.scan[w];
      sm.total_u = tot;
    }
    __syncthreads();
    U = sm.total_u;
    __syncthreads();  // sm.scan is reused by the start search below
    // the launch has a CTA per SM; a step with fewer key blocks uses the first U of
    // them (every CTA of the partition keeps at least one block), the rest have none
    C = decode_ctas_used(U, C);
    if (b >= C) return;  // uniform over the CTA; no pipeline started
  }

  const long long u_lo = (long long)b * U / C;
  const long long u_hi = (long long)(b + 1) * U / C;

  // ---- this CTA's first request: from the host's table, or by a block scan
  if (p.has_table) {
    if (threadIdx.x == 0) {
      sm.first_r = p.cta_first[b].r;
      sm.first_u = p.cta_first[b].u_r;
    }
    __syncthreads();
  } else if (u_lo < u_hi) {
    long long carry = 0;
    for (int base_r = 0; base_r < R; base_r += nthreads) {
      const int r = base_r + threadIdx.x;
      int seq = 0, t = 0, units = 0;
      if (r < R) units = decode_units(p.a, r, &seq, &t);
      long long v = warp_incl_scan(units);
      if (lane == 31) sm.scan[warp] = v;
      __syncthreads();
      if (warp == 0) {
        long long w = lane < (nthreads >> 5) ? sm.scan[lane] : 0;
        w = warp_incl_scan(w);
        if (lane < (nthreads >> 5)) sm.scan[lane] = w;  // inclusive totals per warp
      }
      __syncthreads();
      const long long before = carry + (warp > 0 ? sm.scan[warp - 1] : 0);
      const long long incl = before + v;
      const long long excl = incl - units;
      if (units > 0 && excl <= u_lo && u_lo < incl) {
        sm.first_r = r;
        sm.first_u = excl;
      }
      carry += sm.scan[(nthreads >> 5) - 1];
      __syncthreads();
      if (sm.first_r >= 0) break;
    }
  }
  allow_dependent_launch();

  const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(p.a.q);
  const int q_row_elems = p.a.num_q_heads * D;
  const uint32_t q_bytes = (uint32_t)(HB * G * D * 2);

  // the producer's counts of query segments published and key blocks issued (read by
  // its drain after the CTA's final barrier)
  int prod_k = 0;
  long long prod_i = 0;
  if (warp == HB) {
    // =================================================== producer warp
    // Request metadata is read 32 requests at a time (lane l holds request
    // wbase + l), and the block-table entries of the next batch of 32 key
    // blocks are requested one batch ahead, so segment switches do not stall
    // the TMA issue on global-memory latency.
    int& k = prod_k;        // segments published
    long long& i = prod_i;  // stages issued
    // the KV stream is read once: it leaves L2 first, ahead of the partials that
    // the combine kernel reads back
    const uint64_t kv_policy = l2_policy_evict_first();

    bool ok = true;
    int wbase = -1, w_units = 0, w_seq = 0, w_t = 0;
    auto load_window = [&](int r0) {
      wbase = r0;
      const int r = r0 + lane;
      int seq = 0, t = 0, units = 0;
      if (r < R) units = decode_units(p.a, r, &seq, &t);
      w_units = units;
      w_seq = seq;
      w_t = t;
    };
    // next decode request at or after r (R when none)
    auto next_decode = [&](int r) -> int {
      while (r < R) {
        if (r - wbase >= 32 || r < wbase) load_window(r);
        const unsigned m = __ballot_sync(0xffffffffu, w_units > 0 && wbase + lane >= r);
        if (m) return wbase + __ffs(m) - 1;
        r = wbase + 32;
      }
      return R;
    };
    const bool pages8 = p.a.block_size < kKB;  // 8-key pages: two per key block
    // page id(s) of key block kb_start + lane (lane < n): with 8-key pages the block's
    // second page goes to pg2 (-1 past the request's last page, whose table entry may
    // not exist)
    int pg2_next = -1;
    auto load_pages = [&](int r, int kb_start, int n, int seq_r) -> int {
      int pg = 0;
      pg2_next = -1;
      if (lane < n) {
        const int32_t* row = p.a.block_table + (long long)r * p.a.bt_stride;
        const int lp = (kb_start + lane) * kKB / p.a.block_size;
        pg = __ldg(row + bt_entry(lp, p.a.ring_blocks));
        if (pages8 && (lp + 1) * p.a.block_size < seq_r)
          pg2_next = __ldg(row + bt_entry(lp + 1, p.a.ring_blocks));
      }
      return pg;
    };
    // walk state of the current segment
    int r = -1, seq = 0, t = 0, units = 0;
    long long u_r = 0, u = u_lo;
    auto fetch = [&](int rr) {
      const int j = rr - wbase;
      units = __shfl_sync(0xffffffffu, w_units, j);
      seq = __shfl_sync(0xffffffffu, w_seq, j);
      t = __shfl_sync(0xffffffffu, w_t, j);
    };
    int kb0 = 0, kb1 = 0;
    int pages = 0;  // page ids of the batch about to be issued (lane j: key block kb + j)
    int pages2 = -1;  // 8-key pages: the block's second page
    if (u_lo < u_hi && sm.first_r >= 0) {
      r = sm.first_r;
      u_r = sm.first_u;
      if (p.has_table) {
        // the host placed the first segment: the first copies wait only on its page
        // ids; the window of following requests is needed at the first switch
        const DecodeCtaStart& c = p.cta_first[b];
        kb0 = c.kb0;
        kb1 = c.kb1;
        t = c.t;
        seq = c.seq;
        units = units_of(seq, p.a.sliding_window);
        pages = load_pages(r, kb0, min(32, kb1 - kb0), seq);
        pages2 = pg2_next;
        load_window(r);
      } else {
        load_window(r);
        fetch(r);
        const int kbl = kb_lo_of(seq, p.a.sliding_window);
        kb0 = kbl + (int)(u - u_r);
        kb1 = kbl + (int)(min(u_r + units, u_hi) - u_r);
        pages = load_pages(r, kb0, min(32, kb1 - kb0), seq);
        pages2 = pg2_next;
      }
    }
    if (p.metadata_ready) grid_dependency_wait();  // the scatter must be complete
    while (r >= 0 && ok) {
      const long long seg_u1 = min(u_r + units, u_hi);
      const int b_first = cta_of(u_r, U, C);
      const int b_last = cta_of(u_r + units - 1, U, C);
      const int qs = k & 1;
      if (k >= 2 && !mbar_wait_warp_or_abort(&sm.qempty[qs], ((k >> 1) - 1) & 1, &sm.abort_flag)) {
        ok = false;
        break;
      }
      if (lane == 0) {
        SegDesc& d = sm.seg[qs];
        d.r = r;
        d.kb0 = kb0;
        d.kb1 = kb1;
        d.t = t;
        d.lo = p.a.sliding_window > 0 ? max(0, seq - p.a.sliding_window) : 0;
        d.hi = seq - 1;
        d.slot = r + b;
        d.direct = (b_first == b_last);
        mbar_arrive_expect_tx(&sm.qfull[qs], q_bytes);
        bulk_load(qring + qs * p.q_slot_bytes,
                  q + (long long)t * q_row_elems + (long long)hg * HB * G * D, q_bytes,
                  &sm.qfull[qs]);
      }
      __syncwarp();
      // the segment after this one (looked up once this segment's first copy is out)
      int nr = -2, nkb0 = 0, nkb1 = 0;
      const long long nu_r = u_r + units;
      auto lookup_next = [&]() {
        if (nr != -2) return;
        nr = -1;
        if (seg_u1 < u_hi) {
          nr = next_decode(r + 1);
          if (nr >= R) nr = -1;
        }
      };
      for (int kb_base = kb0; kb_base < kb1 && ok; kb_base += 32) {
        const int nkb = min(32, kb1 - kb_base);
        const int cur = pages, cur2 = pages2;
        for (int j = 0; j < nkb; ++j) {
          const int pg = __shfl_sync(0xffffffffu, cur, j);
          const int pg2 = __shfl_sync(0xffffffffu, cur2, j);
          const int kb = kb_base + j;
          const int s = (int)(i % p.stages);
          if (i >= p.stages && !mbar_wait_warp_or_abort(&sm.empty[s],
                                                        (uint32_t)(((i / p.stages) - 1) & 1),
                                                        &sm.abort_flag)) {
            ok = false;
            break;
          }
          if (*reinterpret_cast<volatile int*>(&sm.abort_flag)) { ok = false; break; }
          if (lane == 0) {
            int pgc = pg;
            if (pg < 0 || pg >= p.a.num_blocks) {
              record_error(p.a.error_word, CB_DEVERR_BLOCK_ID_CODE);
              pgc = p.a.num_blocks;  // TMA reads past the pool as zeros
            }
            const int key0 = pages8 ? 0 : (kb * kKB) % p.a.block_size;
            uint8_t* st = stages + s * p.stage_bytes;
            mbar_arrive_expect_tx(&sm.full[s], (uint32_t)p.stage_bytes);
#pragma unroll
            for (int h = 0; h < kHalves; ++h) {
              tma_load_4d_hint(st + h * box_bytes, &tmap_k, &sm.full[s], h * 64, key0, hg * HB,
                               pgc, kv_policy);
              tma_load_4d_hint(st + (kHalves + h) * box_bytes, &tmap_v, &sm.full[s], h * 64,
                               key0, hg * HB, pgc, kv_policy);
            }
            if (pages8) {
              // the block's keys 8-15: the next page (past the request: zeros; its keys
              // are masked and its V rows zeroed by the consumers)
              int pgc2 = pg2;
              if (pg2 >= p.a.num_blocks) {
                record_error(p.a.error_word, CB_DEVERR_BLOCK_ID_CODE);
                pgc2 = p.a.num_blocks;
              } else if (pg2 < 0) {
                pgc2 = p.a.num_blocks;
              }
              const int half8 = HB * 8 * 128;  // rows (page 1, head, key) start here
#pragma unroll
              for (int h = 0; h < kHalves; ++h) {
                tma_load_4d_hint(st + h * box_bytes + half8, &tmap_k, &sm.full[s], h * 64, 0,
                                 hg * HB, pgc2, kv_policy);
                tma_load_4d_hint(st + (kHalves + h) * box_bytes + half8, &tmap_v, &sm.full[s],
                                 h * 64, 0, hg * HB, pgc2, kv_policy);
              }
            }
          }
          __syncwarp();
          ++i;
          if (j == 0) {
            // page ids of the batch after this one: the rest of this segment, or the
            // next segment's start
            if (kb_base + 32 < kb1) {
              pages = load_pages(r, kb_base + 32, min(32, kb1 - kb_base - 32), seq);
              pages2 = pg2_next;
            } else {
              lookup_next();
              if (nr >= 0) {
                const int jn = nr - wbase;
                const int n_units = __shfl_sync(0xffffffffu, w_units, jn);
                const int n_seq = __shfl_sync(0xffffffffu, w_seq, jn);
                const int nkbl = kb_lo_of(n_seq, p.a.sliding_window);
                nkb0 = nkbl;
                nkb1 = nkbl + (int)(min(nu_r + n_units, u_hi) - nu_r);
                pages = load_pages(nr, nkb0, min(32, nkb1 - nkb0), n_seq);
                pages2 = pg2_next;
              }
            }
          }
        }
      }
      ++k;
      if (!ok) break;
      lookup_next();
      if (nr < 0) break;
      // advance to the next segment
      r = nr;
      u_r = nu_r;
      u = seg_u1;
      fetch(r);
      kb0 = nkb0;
      kb1 = nkb1;
    }
    if (ok) {
      // terminator
      const int qs = k & 1;
      if (k >= 2 && !mbar_wait_warp_or_abort(&sm.qempty[qs], ((k >> 1) - 1) & 1, &sm.abort_flag))
        ok = false;
      if (ok && lane == 0) {
        sm.seg[qs].r = -1;
        mbar_arrive(&sm.qfull[qs]);
      }
    }
    if (!ok && lane == 0) {
      record_error(p.a.error_word, CB_DEVERR_TIMEOUT_CODE);
      set_abort(&sm.abort_flag);
    }
  } else {
  // ===================================================== consumer warps
  // (a lambda, so that a wait that gives up leaves it with a return and still reaches
  // the CTA's final barrier)
  auto consume = [&]() {
  const int hl = warp;  // local KV head
  const bool pages8 = p.a.block_size < kKB;
  constexpr int kRowChunks = D / 8;  // 16-byte chunks of one head's K (or V) row
  const long long num_slots = (long long)p.a.num_blocks * p.a.block_size;
  const int gid = lane >> 2;
  const int tq = lane & 3;
  const float sl2 = p.a.scale_log2;
  long long i = 0;
  if (p.a.test_expire_wait) {
    // test hook: this warp's first wait runs out (nothing arrives at sm.never)
    if (!mbar_wait_warp_polls(&sm.never, 0, kTestExpiryPolls)) {
      if (lane == 0) {
        record_error(p.a.error_word, CB_DEVERR_TIMEOUT_CODE);
        set_abort(&sm.abort_flag);
      }
      return;
    }
  }
  for (int k = 0;; ++k) {
    const int qs = k & 1;
    if (!mbar_wait_warp_or_abort(&sm.qfull[qs], (k >> 1) & 1, &sm.abort_flag)) {
      if (lane == 0) {
        record_error(p.a.error_word, CB_DEVERR_TIMEOUT_CODE);
        set_abort(&sm.abort_flag);
      }
      return;
    }
    const SegDesc d = sm.seg[qs];
    if (d.r < 0) break;
    // fused scatter (steps of decode rows only): the segment holding the request's
    // last key block takes the request's new K/V row of this warp's head -- lane c <
    // kRowChunks: 16-byte chunk c of K, the next kRowChunks lanes the same chunks of V --
    // writes it to the row's cache slot and over the stale copy of that position in the
    // staged block, so no other CTA and no copy engine needs to see the write
    const int kb_last = d.hi / kKB;
    const bool fused_row = p.fuse_scatter && d.kb1 == kb_last + 1;
    long long row_slot = -1;
    uint4 new_row = make_uint4(0u, 0u, 0u, 0u);
    if (fused_row) {
      row_slot = __ldg(p.slot_mapping + d.t);
      if (lane < 2 * kRowChunks) {
        const uint4* src = static_cast<const uint4*>(lane < kRowChunks ? p.k_new : p.v_new);
        new_row = __ldg(src + ((long long)d.t * p.a.num_kv_heads + hg * HB + hl) * kRowChunks +
                        lane % kRowChunks);
      }
    }
    // query fragments (B operand of S^T = K Q^T): Q[head = 8 nb + gid][d = 16ks + 2tq (+8)]
    uint32_t qf[NB][kKSteps][2];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
      const int head = 8 * nb + gid;
      const uint32_t* qrow = reinterpret_cast<const uint32_t*>(qring + qs * p.q_slot_bytes +
                                                               (hl * G + head) * D * 2);
#pragma unroll
      for (int ks = 0; ks < kKSteps; ++ks) {
        qf[nb][ks][0] = head < G ? qrow[(16 * ks + 2 * tq) >> 1] : 0u;
        qf[nb][ks][1] = head < G ? qrow[(16 * ks + 2 * tq + 8) >> 1] : 0u;
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.qempty[qs]);

    float o[NB][kKSteps][4];
    float m0[NB], m1[NB], l0[NB], l1[NB];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
#pragma unroll
      for (int m = 0; m < kKSteps; ++m) o[nb][m][0] = o[nb][m][1] = o[nb][m][2] = o[nb][m][3] = 0.f;
      m0[nb] = m1[nb] = -FLT_MAX;
      l0[nb] = l1[nb] = 0.f;
    }

    for (int kb = d.kb0; kb < d.kb1; ++kb, ++i) {
      const int s = (int)(i % p.stages);
      if (!mbar_wait_warp_or_abort(&sm.full[s], (uint32_t)((i / p.stages) & 1), &sm.abort_flag)) {
        if (lane == 0) {
          record_error(p.a.error_word, CB_DEVERR_TIMEOUT_CODE);
          set_abort(&sm.abort_flag);
        }
        return;
      }
      uint8_t* ks_base = stages + s * p.stage_bytes;
      uint8_t* vs_base = stages + s * p.stage_bytes + kHalves * box_bytes;
      const int key_base = kb * kKB;
      if (fused_row && kb == kb_last) {
        if (row_slot >= 0 && row_slot < num_slots) {
          if (lane < 2 * kRowChunks) {
            const int c = lane % kRowChunks;
            const int key = d.hi - key_base;
            uint8_t* tile = lane < kRowChunks ? ks_base : vs_base;
            *reinterpret_cast<uint4*>(tile + (c >> 3) * box_bytes + stage_row(pages8, HB, hl, key) * 128 +
                                      (((c & 7) ^ (key & 7)) << 4)) = new_row;
            uint4* cache = static_cast<uint4*>(lane < kRowChunks ? p.a.k_cache : p.a.v_cache);
            cache[(row_slot * p.a.num_kv_heads + hg * HB + hl) * kRowChunks + c] = new_row;
            // the producer's next tensor copy into this stage (async proxy) must land
            // after this ordinary store: order it before the stage's release below
            fence_proxy_async_smem();
          }
        } else if (row_slot >= num_slots && lane == 0) {
          record_error(p.a.error_word, CB_DEVERR_SLOT_CODE);
        }
        __syncwarp();
      }
      // zero V rows past the last attended key (their page slots hold unrelated data)
      if (key_base + kKB - 1 > d.hi) {
        const int first_bad = d.hi - key_base + 1;
        const int nbad = kKB - first_bad;
        for (int e = lane; e < nbad * kHalves * 8; e += 32) {
          const int row = first_bad + e / (kHalves * 8);
          const int rem = e % (kHalves * 8);
          const int h = rem >> 3;
          const int c = rem & 7;
          *reinterpret_cast<uint4*>(vs_base + h * box_bytes + stage_row(pages8, HB, hl, row) * 128 +
                                    c * 16) = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();  // as above: before the stage is handed back to the copies
        __syncwarp();
      }
      // ---- S^T = K Q^T  (16 keys x 8 heads per column block)
      float sacc[NB][4];
#pragma unroll
      for (int nb = 0; nb < NB; ++nb) sacc[nb][0] = sacc[nb][1] = sacc[nb][2] = sacc[nb][3] = 0.f;
      {
        const int jm = lane >> 3;
        const int key = (lane & 7) + ((jm & 1) << 3);
        const uint32_t row_addr = smem_u32(ks_base) + stage_row(pages8, HB, hl, key) * 128;
#pragma unroll
        for (int ks = 0; ks < kKSteps; ++ks) {
          const int chunk = (ks & 3) * 2 + (jm >> 1);
          uint32_t a[4];
          ldmatrix_x4(a, row_addr + (ks >> 2) * box_bytes + ((chunk ^ (key & 7)) << 4));
#pragma unroll
          for (int nb = 0; nb < NB; ++nb) mma_bf16_16816(sacc[nb], a, qf[nb][ks][0], qf[nb][ks][1]);
        }
      }
      // ---- mask, online softmax per head column (8 nb + 2tq, 8 nb + 2tq + 1)
      const int k0 = key_base + gid;
      const int k1 = k0 + 8;
      const bool v0 = k0 >= d.lo && k0 <= d.hi;
      const bool v1 = k1 >= d.lo && k1 <= d.hi;
      uint32_t pb0[NB], pb1[NB];
#pragma unroll
      for (int nb = 0; nb < NB; ++nb) {
        const float s0 = v0 ? sacc[nb][0] * sl2 : -INFINITY;
        const float s1 = v0 ? sacc[nb][1] * sl2 : -INFINITY;
        const float s2 = v1 ? sacc[nb][2] * sl2 : -INFINITY;
        const float s3 = v1 ? sacc[nb][3] * sl2 : -INFINITY;
        float mx0 = fmaxf(s0, s2), mx1 = fmaxf(s1, s3);
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
          mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
          mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
        }
        const float mn0 = fmaxf(m0[nb], mx0), mn1 = fmaxf(m1[nb], mx1);
        const float a0 = exp2f(m0[nb] - mn0), a1 = exp2f(m1[nb] - mn1);
        const float p0 = exp2f(s0 - mn0), p1 = exp2f(s1 - mn1);
        const float p2 = exp2f(s2 - mn0), p3 = exp2f(s3 - mn1);
        m0[nb] = mn0;
        m1[nb] = mn1;
        l0[nb] = l0[nb] * a0 + (p0 + p2);
        l1[nb] = l1[nb] * a1 + (p1 + p3);
#pragma unroll
        for (int m = 0; m < kKSteps; ++m) {
          o[nb][m][0] *= a0;
          o[nb][m][1] *= a1;
          o[nb][m][2] *= a0;
          o[nb][m][3] *= a1;
        }
        pb0[nb] = movmatrix_trans(pack_bf16x2(p0, p1));  // keys 0-7
        pb1[nb] = movmatrix_trans(pack_bf16x2(p2, p3));  // keys 8-15
      }
      // ---- O^T += V^T P^T  (D x 8 heads per column block)
      {
        const int jm = lane >> 3;
        const int key = (lane & 7) + ((jm >> 1) << 3);
        const uint32_t row_addr = smem_u32(vs_base) + stage_row(pages8, HB, hl, key) * 128;
#pragma unroll
        for (int m = 0; m < kKSteps; ++m) {
          const int chunk = 2 * m + (jm & 1);
          uint32_t a[4];
          ldmatrix_x4_trans(a, row_addr + (chunk >> 3) * box_bytes +
                                   (((chunk & 7) ^ (key & 7)) << 4));
#pragma unroll
          for (int nb = 0; nb < NB; ++nb) mma_bf16_16816(o[nb][m], a, pb0[nb], pb1[nb]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.empty[s]);
    }

    // ---- segment epilogue
    const int qh_base = (hg * HB + hl) * G;
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
      float sl0 = l0[nb], sl1 = l1[nb];
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        sl0 += __shfl_xor_sync(0xffffffffu, sl0, off);
        sl1 += __shfl_xor_sync(0xffffffffu, sl1, off);
      }
      const int h0 = 8 * nb + 2 * tq, h1 = h0 + 1;
      if (d.direct) {
        __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.a.out) + (long long)d.t * q_row_elems;
        const float i0 = 1.f / sl0, i1 = 1.f / sl1;
#pragma unroll
        for (int m = 0; m < kKSteps; ++m) {
          const int dd = 16 * m + gid;
          if (h0 < G) {
            out[(qh_base + h0) * D + dd] = __float2bfloat16_rn(o[nb][m][0] * i0);
            out[(qh_base + h0) * D + dd + 8] = __float2bfloat16_rn(o[nb][m][2] * i0);
          }
          if (h1 < G) {
            out[(qh_base + h1) * D + dd] = __float2bfloat16_rn(o[nb][m][1] * i1);
            out[(qh_base + h1) * D + dd + 8] = __float2bfloat16_rn(o[nb][m][3] * i1);
          }
        }
      } else {
        float* po = p.part_o + (long long)d.slot * q_row_elems;
#pragma unroll
        for (int m = 0; m < kKSteps; ++m) {
          const int dd = 16 * m + gid;
          if (h0 < G) {
            po[(qh_base + h0) * D + dd] = o[nb][m][0];
            po[(qh_base + h0) * D + dd + 8] = o[nb][m][2];
          }
          if (h1 < G) {
            po[(qh_base + h1) * D + dd] = o[nb][m][1];
            po[(qh_base + h1) * D + dd + 8] = o[nb][m][3];
          }
        }
        if (gid == 0) {
          float2* pml = p.part_ml + (long long)d.slot * p.a.num_q_heads;
          if (h0 < G) pml[qh_base + h0] = make_float2(m0[nb], sl0);
          if (h1 < G) pml[qh_base + h1] = make_float2(m1[nb], sl1);
        }
      }
    }
  }
  };
  consume();
  }

  // Every warp has stopped issuing and waiting. If a wait gave up somewhere in the CTA,
  // copies the producer issued may not have been consumed: each stage slot and each
  // query slot has at most one copy in flight, the latest issued into it (a slot is
  // refilled only after its previous copy was consumed), so waiting for the phase of
  // the latest copy of each slot drains them all before the shared memory is released.
  __syncthreads();
  if (warp == HB && lane == 0 && *reinterpret_cast<volatile int*>(&sm.abort_flag)) {
    const long long first = prod_i > p.stages ? prod_i - p.stages : 0;
    for (long long j = first; j < prod_i; ++j)
      mbar_wait(&sm.full[j % p.stages], (uint32_t)((j / p.stages) & 1));
    for (int seg = prod_k > 2 ? prod_k - 2 : 0; seg < prod_k; ++seg)
      mbar_wait(&sm.qfull[seg & 1], (uint32_t)((seg >> 1) & 1));
  }
}

// Combine of the split decode requests: out = sum_s 2^(m_s - M) o_s /
// sum_s 2^(m_s - M) l_s over the request's segments s (M = max_s m_s), the
// log-sum-exp merge of split-KV partials. CTA (x, y) takes request x of the
// host's list (or, with no list, request x itself, found split or not by the
// same partition arithmetic as the decode grid) and KV heads
// [y * kv_per_cta, (y + 1) * kv_per_cta): one thread per four consecutive
// outputs, the partials of up to twelve segments in flight per thread. The host
// sizes the grid to about one CTA per SM, so a request split over ten CTAs is
// merged on several SMs at once. The kernel is launched right after the decode
// kernel and waits for it on the device (programmatic dependent launch), with
// its list entry or scan already done.
template <int D, int G>
__global__ void __launch_bounds__(kCombineMaxThreads)
decode_combine_kernel(const CombineArgs c) {
  constexpr int kChunk = kCombineSegmentsInFlight;
  __shared__ long long red[32];
  __shared__ long long totals[2];
  const int x = blockIdx.x;
  const int kvh0 = blockIdx.y * c.kv_per_cta;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int nthreads = blockDim.x;
  allow_dependent_launch();
  int r, t, b_first, nseg;
  if (c.n_entries >= 0) {
    if (x >= c.n_entries) return;
    const CombineEntry e = c.entries[x];
    r = e.r;
    t = e.t;
    b_first = e.b_first;
    nseg = e.nseg;
  } else {
    // the decode grid's partition from the device metadata: U (all decode key
    // blocks), the key blocks of the requests before x, and C (CTAs in use)
    const StepArgs& a = c.a;
    r = x;
    if (r >= a.num_requests) return;
    long long all = 0, before = 0;
    for (int i = threadIdx.x; i < a.num_requests; i += nthreads) {
      int sq = 0, tt = 0;
      const int u = decode_units(a, i, &sq, &tt);
      all += u;
      if (i < r) before += u;
    }
    for (int k = 0; k < 2; ++k) {
      long long v = k == 0 ? all : before;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
      if (lane == 0) red[warp] = v;
      __syncthreads();
      if (threadIdx.x == 0) {
        long long tot = 0;
        for (int w = 0; w < (nthreads >> 5); ++w) tot += red[w];
        totals[k] = tot;
      }
      __syncthreads();
    }
    int seq = 0;
    const int units = decode_units(a, r, &seq, &t);
    const long long U = totals[0];
    if (units == 0 || U == 0) return;
    const int C = decode_ctas_used(U, c.num_ctas);
    b_first = cta_of(totals[1], U, C);
    nseg = cta_of(totals[1] + units - 1, U, C) - b_first + 1;
    if (nseg < 2) return;  // written directly by its CTA
  }
  // thread (part, f): float4 f of the slice (outputs 4f .. 4f + 3) over segment range
  // `part` of the request's; the partitions' results are merged through shared memory
  const int F = c.kv_per_cta * G * D / 4;
  const int nparts = c.parts;
  const int f = threadIdx.x % F;
  const int part = threadIdx.x / F;
  const int Hq = c.a.num_q_heads;
  const int qh = kvh0 * G + (4 * f) / D;
  const long long slot0 = (long long)r + b_first;
  const int o_off = kvh0 * G * D / 4 + f;  // float4 index within a slot
  // segment s: ml_base[s * Hq], o_base[s * o_stride]
  const float2* ml_base = c.part_ml + slot0 * Hq + qh;
  const float4* o_base = reinterpret_cast<const float4*>(c.part_o + slot0 * Hq * D) + o_off;
  const int o_stride = Hq * D / 4;
  const int s_begin = part * nseg / nparts, s_end = (part + 1) * nseg / nparts;
  // the partials of CTAs that finished early may have left L2: ask for them while
  // the decode grid drains (a hint; the values are read after the wait)
  for (int i = s_begin; i < s_end; ++i) {
    if ((4 * f) % D == 0) prefetch_l2(ml_base + i * Hq);
    if (f % 8 == 0) prefetch_l2(o_base + (long long)i * o_stride);
  }
  grid_dependency_wait();  // the partials of the decode grid
  float M = -FLT_MAX, L = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s0 = s_begin; s0 < s_end; s0 += kChunk) {
    const int n = min(kChunk, s_end - s0);
    float2 ml[kChunk];
    float4 o[kChunk];
#pragma unroll
    for (int i = 0; i < kChunk; ++i) {
      if (i < n) {
        ml[i] = __ldcg(ml_base + (s0 + i) * Hq);
        o[i] = __ldcg(o_base + (long long)(s0 + i) * o_stride);
      }
    }
    float mb = M;
#pragma unroll
    for (int i = 0; i < kChunk; ++i)
      if (i < n) mb = fmaxf(mb, ml[i].x);
    const float sc = exp2f(M - mb);  // 0 on the first chunk (acc and L are 0 then)
    M = mb;
    L *= sc;
    acc.x *= sc;
    acc.y *= sc;
    acc.z *= sc;
    acc.w *= sc;
#pragma unroll
    for (int i = 0; i < kChunk; ++i) {
      if (i < n) {
        const float w = exp2f(ml[i].x - mb);
        L = fmaf(w, ml[i].y, L);
        acc.x = fmaf(w, o[i].x, acc.x);
        acc.y = fmaf(w, o[i].y, acc.y);
        acc.z = fmaf(w, o[i].z, acc.z);
        acc.w = fmaf(w, o[i].w, acc.w);
      }
    }
  }
  if (nparts > 1) {
    extern __shared__ float4 red_acc[];  // [nparts * F], then red_ml
    float2* red_ml = reinterpret_cast<float2*>(red_acc + nparts * F);
    red_acc[threadIdx.x] = acc;
    red_ml[threadIdx.x] = make_float2(M, L);
    __syncthreads();
    if (part != 0) return;
    for (int q = 1; q < nparts; ++q) M = fmaxf(M, red_ml[q * F + f].x);
    L = 0.f;
    acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int q = 0; q < nparts; ++q) {
      const float2 ml = red_ml[q * F + f];
      const float4 o = red_acc[q * F + f];
      const float w = exp2f(ml.x - M);  // 0 for a partition without segments
      L = fmaf(w, ml.y, L);
      acc.x = fmaf(w, o.x, acc.x);
      acc.y = fmaf(w, o.y, acc.y);
      acc.z = fmaf(w, o.z, acc.z);
      acc.w = fmaf(w, o.w, acc.w);
    }
  }
  const float inv = 1.f / L;
  uint2 packed;
  packed.x = pack_bf16x2(acc.x * inv, acc.y * inv);
  packed.y = pack_bf16x2(acc.z * inv, acc.w * inv);
  __nv_bfloat16* out = static_cast<__nv_bfloat16*>(c.a.out) + (long long)t * Hq * D;
  reinterpret_cast<uint2*>(out)[o_off] = packed;
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

// 4-D view of a cache [NB, BS, Hkv, D] as (d, key-in-page, head, page) so that
// a box (64, 16, HB, 1) lands in shared memory head-major: rows (head, key).
cudaError_t make_cache_map(CUtensorMap* map, void* cache, const StepArgs& a, int hb) {
  auto fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  const cuuint64_t elt = 2;
  cuuint64_t dims[4] = {(cuuint64_t)a.head_dim, (cuuint64_t)a.block_size,
                        (cuuint64_t)a.num_kv_heads, (cuuint64_t)a.num_blocks};
  cuuint64_t strides[3] = {(cuuint64_t)a.num_kv_heads * a.head_dim * elt,
                           (cuuint64_t)a.head_dim * elt,
                           (cuuint64_t)a.block_size * a.num_kv_heads * a.head_dim * elt};
  // 16 keys of one page, or all 8 of an 8-key page (a block then takes two boxes)
  cuuint32_t box[4] = {64, (cuuint32_t)(a.block_size < 16 ? a.block_size : 16), (cuuint32_t)hb, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, cache, dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int D, int G>
cudaError_t launch_dg(const DecodeArgs& p, const CUtensorMap& mk, const CUtensorMap& mv,
                      size_t smem, int hg, int num_requests, cudaStream_t s) {
  auto kern = decode_split_kernel<D, G>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kDecodeSmemLimit);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  (void)num_requests;
  return launch_pdl(kDecodeSplit, kern, dim3(p.num_ctas, hg), dim3(p.heads_per_cta * 32 + 32),
                    smem, s, mk, mv, p);
}

template <int D>
cudaError_t launch_d(const DecodeArgs& p, const CUtensorMap& mk, const CUtensorMap& mv,
                     size_t smem, int hg, int R, cudaStream_t s) {
  switch (p.a.num_q_heads / p.a.num_kv_heads) {
    case 1: return launch_dg<D, 1>(p, mk, mv, smem, hg, R, s);
    case 2: return launch_dg<D, 2>(p, mk, mv, smem, hg, R, s);
    case 4: return launch_dg<D, 4>(p, mk, mv, smem, hg, R, s);
    case 8: return launch_dg<D, 8>(p, mk, mv, smem, hg, R, s);
    case 16: return launch_dg<D, 16>(p, mk, mv, smem, hg, R, s);
  }
  return cudaErrorInvalidValue;
}

template <int D>
cudaError_t launch_combine_d(const CombineArgs& c, dim3 grid, dim3 block, size_t smem,
                             cudaStream_t s) {
  switch (c.a.num_q_heads / c.a.num_kv_heads) {
    case 1: return launch_pdl(kDecodeCombine, decode_combine_kernel<D, 1>, grid, block, smem, s, c);
    case 2: return launch_pdl(kDecodeCombine, decode_combine_kernel<D, 2>, grid, block, smem, s, c);
    case 4: return launch_pdl(kDecodeCombine, decode_combine_kernel<D, 4>, grid, block, smem, s, c);
    case 8: return launch_pdl(kDecodeCombine, decode_combine_kernel<D, 8>, grid, block, smem, s, c);
    case 16: return launch_pdl(kDecodeCombine, decode_combine_kernel<D, 16>, grid, block, smem, s, c);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_decode_combine(const CombineArgs& c, cudaStream_t stream) {
  const int nx = c.n_entries >= 0 ? c.n_entries : c.a.num_requests;
  if (nx <= 0) return cudaSuccess;
  const int G = c.a.num_q_heads / c.a.num_kv_heads;
  const int f4 = c.kv_per_cta * G * c.a.head_dim / 4;
  if (c.kv_per_cta <= 0 || c.a.num_kv_heads % c.kv_per_cta != 0 || f4 > kCombineMaxThreads)
    return cudaErrorInvalidValue;
  const dim3 grid(nx, c.a.num_kv_heads / c.kv_per_cta);
  if (c.parts < 1 || f4 * c.parts > kCombineMaxThreads) return cudaErrorInvalidValue;
  // f4 = kv_per_cta x G x D / 4 is a multiple of 32
  const dim3 block(f4 * c.parts);
  const size_t smem = c.parts > 1 ? (size_t)block.x * (sizeof(float4) + sizeof(float2)) : 0;
  if (c.a.head_dim == 64) return launch_combine_d<64>(c, grid, block, smem, stream);
  return launch_combine_d<128>(c, grid, block, smem, stream);
}

size_t decode_smem_bytes(int stages, int stage_bytes, int q_slot_bytes) {
  return 1024 /* alignment slack */ + (size_t)stages * stage_bytes + 2 * (size_t)q_slot_bytes +
         sizeof(DecodeSmem);
}

cudaError_t prepare_decode(const DecodeArgs& p) {
  const int G = p.a.num_q_heads / p.a.num_kv_heads;
  auto set = [](auto kern) {
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kDecodeSmemLimit);
  };
  if (p.a.head_dim == 64) {
    switch (G) {
      case 1: return set(decode_split_kernel<64, 1>);
      case 2: return set(decode_split_kernel<64, 2>);
      case 4: return set(decode_split_kernel<64, 4>);
      case 8: return set(decode_split_kernel<64, 8>);
      case 16: return set(decode_split_kernel<64, 16>);
    }
  } else {
    switch (G) {
      case 1: return set(decode_split_kernel<128, 1>);
      case 2: return set(decode_split_kernel<128, 2>);
      case 4: return set(decode_split_kernel<128, 4>);
      case 8: return set(decode_split_kernel<128, 8>);
      case 16: return set(decode_split_kernel<128, 16>);
    }
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_decode(DecodeArgs p, const DecodePlan& plan, cudaStream_t stream) {
  CUtensorMap mk, mv;
  cudaError_t e = make_cache_map(&mk, p.a.k_cache, p.a, p.heads_per_cta);
  if (e == cudaSuccess) e = make_cache_map(&mv, p.a.v_cache, p.a, p.heads_per_cta);
  if (e != cudaSuccess) return e;
  const int hg = p.a.num_kv_heads / p.heads_per_cta;
  if (p.a.head_dim == 64) return launch_d<64>(p, mk, mv, plan.smem_bytes, hg, p.a.num_requests, stream);
  return launch_d<128>(p, mk, mv, plan.smem_bytes, hg, p.a.num_requests, stream);
}

}  // namespace cb
