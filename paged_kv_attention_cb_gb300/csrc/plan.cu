// Host-side planning of one step from the host mirrors of the metadata. The
// scheduler metadata "already divides the work into a request's query tile /
// KV tile" ("Continuous Batching", languisher.top, section "Extension: the
// vLLM v1 implementation"); here that division is made per call: decode rows
// go to the split-KV kernel with a byte-balanced partition, prefill rows to
// the prefill kernel, and whatever the fast kernels do not cover to the
// portable kernel.
#include <stdlib.h>

#include <algorithm>
#include <utility>
#include <vector>

#include "cb.h"
#include "decode.h"
#include "plan.h"

namespace cb {

namespace {

constexpr size_t align256(size_t x) { return (x + 255) & ~size_t(255); }
constexpr int kRowsPerTile = 128;  // query rows (tokens x grouped heads) per prefill tile

int sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (!cached[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    cached[dev] = n;
  }
  return cached[dev];
}

struct WorkspaceLayout {
  size_t part_ml, part_o, total;
};

WorkspaceLayout layout(int32_t R, int32_t Hq, int32_t Hkv, int32_t D) {
  (void)Hkv;
  WorkspaceLayout w;
  const size_t slots = (size_t)std::max(R, 0) + kMaxDecodeCtas;
  w.part_ml = kWorkspaceHeaderBytes;
  w.part_o = w.part_ml + align256(slots * Hq * 8);
  w.total = w.part_o + slots * Hq * (size_t)D * 4;
  return w;
}

// The layout of a workspace of `bytes`: that of the largest request count it holds,
// not of the step's own count, so that every step on one workspace finds the
// partial (m, l) and the partial outputs at the same offsets. The estimate is
// conservative: layout(R).total <= bytes.
WorkspaceLayout layout_of(size_t bytes, const StepArgs& a) {
  const size_t Hq = (size_t)a.num_q_heads, D = (size_t)a.head_dim;
  const size_t per_request = Hq * 8 + Hq * D * 4;
  const size_t fixed = kWorkspaceHeaderBytes + 512 + (size_t)kMaxDecodeCtas * (Hq * 8 + Hq * D * 4);
  long long r = bytes > fixed ? (long long)((bytes - fixed) / per_request) : 0;
  r = std::min<long long>(r, 1 << 24);
  r = std::max<long long>(r, a.num_requests);  // the size check left room for the step's R
  return layout((int32_t)r, a.num_q_heads, a.num_kv_heads, a.head_dim);
}

// First key block (16 keys) a decode query attends, and the number of blocks it attends.
int kb_lo_host(int seq, int window) { return (window > 0 ? std::max(0, seq - window) : 0) / 16; }

int decode_units_host(int seq, int window) { return (seq - 1) / 16 - kb_lo_host(seq, window) + 1; }

// CTA of the decode partition that owns global key block u (ranges [b U/C, (b+1) U/C)).
int cta_of_host(long long u, long long U, int C) { return (int)(((u + 1) * C + U - 1) / U) - 1; }

void combine_common(CombineArgs& c, const StepArgs& a, const DecodeArgs& d) {
  c.a = a;
  c.num_ctas = d.num_ctas;
  c.part_o = d.part_o;
  c.part_ml = d.part_ml;
}

// KV heads per combine CTA for `n` requests to merge: the fewest (most CTAs) that
// keep the grid within about one CTA per SM, a divisor of Hkv, and at most
// kCombineMaxThreads threads (four outputs each) per CTA.
int combine_kv_per_cta(const StepArgs& a, int n) {
  const int Hkv = a.num_kv_heads, G = a.num_q_heads / a.num_kv_heads;
  int best = 0;
  for (int k = Hkv; k >= 1; --k) {
    if (Hkv % k != 0 || k * G * a.head_dim / 4 > kCombineMaxThreads) continue;
    if (best == 0 || (long long)std::max(n, 1) * (Hkv / k) <= sm_count()) best = k;
  }
  return best;
}

}  // namespace

size_t workspace_bytes(int32_t num_requests, int32_t num_tokens, int32_t num_q_heads,
                       int32_t num_kv_heads, int32_t head_dim) {
  (void)num_tokens;
  if (num_requests < 0 || num_q_heads <= 0 || head_dim <= 0) return kWorkspaceHeaderBytes;
  return layout(num_requests, num_q_heads, num_kv_heads, head_dim).total;
}

// SMs left to the prefill kernel while the decode kernel streams (concurrent mixed
// step). Model, from measurements of the two kernels side by side on GB300: the decode
// stream runs at min(HBM, C x per-SM rate) on its C SMs; the prefill tiles run at a
// fixed rate per SM, on k SMs until the decode grid finishes and on every SM after
// that. The share minimises the modelled step time (ties: more SMs for the decode).
// CB_PREFILL_SMS overrides it (for measurements).
int prefill_sm_share(long long decode_bytes, double prefill_flops, int n_prefill_ctas, int S) {
  const int kmax = std::max(1, std::min(n_prefill_ctas, S - 1));
  const char* env = getenv("CB_PREFILL_SMS");
  if (env != nullptr && *env != '\0') return std::max(1, std::min(atoi(env), kmax));
  constexpr double kHbm = 6.6e12;          // B/s, decode stream on enough SMs
  constexpr double kHbmPerSm = 75e9;       // B/s, decode stream per SM
  constexpr double kFlopsPerSm = 7.0e12;   // causal-pair FLOP/s of prefill tiles per SM
  int best_k = 1;
  double best_t = 1e30;
  for (int k = 1; k <= kmax; ++k) {
    const double td = (double)decode_bytes / std::min(kHbm, (S - k) * kHbmPerSm);
    const double done = k * kFlopsPerSm * td;  // prefill work finished beside the decode
    const double t = done >= prefill_flops ? std::max(td, prefill_flops / (k * kFlopsPerSm))
                                           : td + (prefill_flops - done) / (S * kFlopsPerSm);
    if (t < best_t * (1.0 - 1e-9)) {
      best_t = t;
      best_k = k;
    }
  }
  return best_k;
}

void plan_step(Plan& plan, const StepArgs& a, const int32_t* h_qsl, const int32_t* h_seq_lens,
               uint32_t flags, const ScatterInputs* scatter, void* workspace,
               size_t workspace_bytes) {
  plan.workspace = workspace;
  plan.workspace_bytes = workspace_bytes;
  plan.fast_decode = false;
  plan.fast_prefill = false;
  plan.n_prefill_launches = 0;
  plan.portable_mode = 0;
  plan.has_combine = false;
  plan.fused_scatter = false;
  plan.concurrent = false;
  if ((flags & CB_FLAG_PORTABLE_ONLY) || a.dtype == CB_F32) return;

  // ---- which rows exist
  long long U = 0;
  bool has_prefill = false;
  double flops = 0.0;  // prefill: causal (query, key) pairs x 4 Hq D
  for (int r = 0; r < a.num_requests; ++r) {
    const int ql = h_qsl[r + 1] - h_qsl[r];
    if (ql == 1 && h_seq_lens[r] > 0) {
      U += decode_units_host(h_seq_lens[r], a.sliding_window);
    } else if (ql > 1) {
      has_prefill = true;
      const long long ctx = h_seq_lens[r] - ql;
      long long pairs = 0;
      if (a.sliding_window > 0) {
        for (int i = 0; i < ql; ++i) pairs += std::min<long long>(ctx + i + 1, a.sliding_window);
      } else {
        pairs = (long long)ql * ctx + (long long)ql * (ql + 1) / 2;
      }
      flops += 4.0 * a.num_q_heads * a.head_dim * (double)pairs;
    }
  }

  // ---- which kernels can take them
  const int G = a.num_q_heads / a.num_kv_heads;
  const int HB = std::min(a.num_kv_heads, kDecodeMaxHeads);
  const bool decode_ok = U > 0 && (a.block_size % 16 == 0 || a.block_size == 8) && G <= 16 &&
                         a.num_kv_heads % HB == 0;
  // a 128-key tile is made of whole page boxes (block_size divides 128) or lies
  // inside one page (block_size a multiple of 128)
  const bool tile_pages_ok = a.block_size % 8 == 0 && (128 % a.block_size == 0 || a.block_size % 128 == 0);
  std::vector<std::pair<long long, int>> order;  // prefill requests (weight, r), heaviest first
  if (has_prefill && tile_pages_ok && G <= 16 && kRowsPerTile % G == 0) {
    for (int r = 0; r < a.num_requests; ++r) {
      const int ql = h_qsl[r + 1] - h_qsl[r];
      if (ql > 1) order.emplace_back(-(long long)h_seq_lens[r] * ql, r);
    }
    std::stable_sort(order.begin(), order.end());
  }
  const int n_launch = (int)((order.size() + kPrefillMaxEntries - 1) / kPrefillMaxEntries);
  const bool prefill_ok = !order.empty() && n_launch <= kMaxPrefillLaunches;
  DecodeArgs& d = plan.decode;
  if (decode_ok) {
    d.stage_bytes = 2 * (a.head_dim / 64) * HB * 16 * 128;
    d.q_slot_bytes = HB * G * a.head_dim * 2;
    const size_t fixed = decode_smem_bytes(0, d.stage_bytes, d.q_slot_bytes);
    d.stages = (int)std::min<size_t>(kDecodeMaxStages, (kDecodeSmemLimit - fixed) / d.stage_bytes);
    plan.fast_decode = d.stages >= 2;
  }
  plan.fast_prefill = prefill_ok;
  if (plan.fast_decode && plan.fast_prefill) plan.portable_mode = -1;
  else if (plan.fast_decode) plan.portable_mode = has_prefill ? 2 : -1;
  else if (plan.fast_prefill) plan.portable_mode = U > 0 ? 1 : -1;
  // Every row on a tensor-core kernel (one prefill launch at most): the kernels write the
  // step's new rows themselves and read the step's own positions from k_new / v_new, so
  // there is no scatter launch; a step with both kinds of rows runs the prefill grid
  // beside the decode grid, on the SMs the decode grid leaves.
  plan.fused_scatter = scatter != nullptr && plan.portable_mode == -1 && n_launch <= 1;
  plan.concurrent = plan.fused_scatter && plan.fast_decode && plan.fast_prefill;
  const bool scatter_first = scatter != nullptr && !plan.fused_scatter;

  // ---- prefill rows: tcgen05 tile kernel, heaviest requests first
  int prefill_total_ctas = 0;
  if (plan.fast_prefill) {
    const int TQ = kRowsPerTile / G;
    for (int l = 0; l < n_launch; ++l) {
      PrefillArgs& pa = plan.prefill[l];
      pa.a = a;
      pa.tile_tokens = TQ;
      pa.box_keys = std::min(a.block_size, 128);
      pa.n_entries = 0;
      // the scatter, the decode kernel or an earlier prefill launch runs first
      pa.metadata_ready = (scatter_first || plan.fast_decode || l > 0) ? 1 : 0;
      pa.device_work = 0;
      pa.total_ctas = 0;
      pa.k_new = plan.fused_scatter ? scatter->k_new : nullptr;
      pa.v_new = plan.fused_scatter ? scatter->v_new : nullptr;
      pa.slot_mapping = plan.fused_scatter ? scatter->slot_mapping : nullptr;
      pa.concurrent = plan.concurrent ? 1 : 0;
      pa.exit_counter = reinterpret_cast<int*>(static_cast<uint8_t*>(workspace) + kExitCounterOffset);
      pa.unit_counter = reinterpret_cast<int*>(static_cast<uint8_t*>(workspace) + kUnitCounterOffset);
      pa.scatter_counter =
          reinterpret_cast<int*>(static_cast<uint8_t*>(workspace) + kScatterCounterOffset);
      for (size_t i = (size_t)l * kPrefillMaxEntries;
           i < order.size() && pa.n_entries < kPrefillMaxEntries; ++i) {
        const int r = order[i].second;
        const int ql = h_qsl[r + 1] - h_qsl[r];
        PrefillEntry& e = pa.entries[pa.n_entries++];
        e.r = r;
        e.n_qtiles = (ql + TQ - 1) / TQ;
        e.q_start = h_qsl[r];
        e.q_len = ql;
        e.seq_len = h_seq_lens[r];
        pa.total_ctas += prefill_ctas(e.n_qtiles, a.num_kv_heads);
      }
      // persistent CTAs, one per SM at most, claim the units heaviest first
      pa.total_units = pa.total_ctas;
      pa.grid = std::min(pa.total_units, sm_count());
      prefill_total_ctas += pa.total_ctas;
    }
    plan.n_prefill_launches = n_launch;
  }

  // ---- decode rows: split-KV kernel
  if (plan.fast_decode) {
    d.a = a;
    d.heads_per_cta = HB;
    d.total_units = U;
    int C = std::min(sm_count(), kMaxDecodeCtas);
    if (plan.concurrent) {
      const long long bytes = U * 16LL * 2 * a.num_kv_heads * a.head_dim * 2;
      C = sm_count() - prefill_sm_share(bytes, flops, prefill_total_ctas, sm_count());
    }
    // at least kDecodeMinBlocksPerCta key blocks per CTA: a small step split over every
    // SM spends more on merging its many segments than it gains in streaming
    d.num_ctas = (int)std::min<long long>(C, (U + kDecodeMinBlocksPerCta - 1) / kDecodeMinBlocksPerCta);
    d.units_on_device = 0;
    // each decode row's new K/V is written by the CTA that reads the request's last key
    // block (the decode kernel is then the step's first)
    d.fuse_scatter = plan.fused_scatter ? 1 : 0;
    d.k_new = scatter ? scatter->k_new : nullptr;
    d.v_new = scatter ? scatter->v_new : nullptr;
    d.slot_mapping = scatter ? scatter->slot_mapping : nullptr;
    d.metadata_ready = scatter_first ? 1 : 0;
    // where each CTA's range [b*U/C, (b+1)*U/C) starts: (request, its first unit)
    d.has_table = d.num_ctas <= kDecodeTableCtas;
    if (d.has_table) {
      long long u = 0;
      int b = 0;
      const long long Cn = d.num_ctas;
      for (int r = 0; r < a.num_requests && b < d.num_ctas; ++r) {
        const int ql = h_qsl[r + 1] - h_qsl[r];
        if (ql != 1 || h_seq_lens[r] <= 0) continue;
        const int units = decode_units_host(h_seq_lens[r], a.sliding_window);
        const int kbl = kb_lo_host(h_seq_lens[r], a.sliding_window);
        while (b < d.num_ctas && (long long)b * U / Cn < u + units) {
          const long long lo = (long long)b * U / Cn, hi = (long long)(b + 1) * U / Cn;
          d.cta_first[b] = DecodeCtaStart{r, (int)u, kbl + (int)(lo - u),
                                          kbl + (int)(std::min(u + units, hi) - u), h_qsl[r],
                                          h_seq_lens[r]};
          ++b;
        }
        u += units;
      }
      for (; b < d.num_ctas; ++b) d.cta_first[b] = DecodeCtaStart{-1, 0, 0, 0, 0, 0};
    }
    const WorkspaceLayout w = layout_of(workspace_bytes, a);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    d.part_ml = reinterpret_cast<float2*>(ws + w.part_ml);
    d.part_o = reinterpret_cast<float*>(ws + w.part_o);
    plan.decode_plan.smem_bytes = decode_smem_bytes(d.stages, d.stage_bytes, d.q_slot_bytes);
    // the requests split over several CTAs, merged by the combine launch
    CombineArgs& c = plan.combine;
    combine_common(c, a, d);
    c.n_entries = 0;
    long long u = 0;
    for (int r = 0; r < a.num_requests; ++r) {
      const int ql = h_qsl[r + 1] - h_qsl[r];
      if (ql != 1 || h_seq_lens[r] <= 0) continue;
      const int units = decode_units_host(h_seq_lens[r], a.sliding_window);
      const int b0 = cta_of_host(u, U, d.num_ctas);
      const int b1 = cta_of_host(u + units - 1, U, d.num_ctas);
      u += units;
      if (b1 == b0) continue;
      if (c.n_entries == kCombineListMax) {
        c.n_entries = -1;  // too many to list: the kernel finds them
        break;
      }
      c.entries[c.n_entries++] = CombineEntry{r, h_qsl[r], b0, b1 - b0 + 1};
    }
    c.kv_per_cta = combine_kv_per_cta(a, c.n_entries >= 0 ? c.n_entries : a.num_requests);
    // a request split into many segments is merged by several threads per output, each
    // over a share of the segments (fewer dependent rounds of loads)
    int max_seg = 0;
    for (int e = 0; e < c.n_entries; ++e) max_seg = std::max(max_seg, c.entries[e].nseg);
    const int f4 = c.kv_per_cta * G * a.head_dim / 4;
    c.parts = max_seg > 2 * kCombineSegmentsInFlight ? std::max(1, kCombineMaxThreads / f4) : 1;
    plan.has_combine = c.n_entries != 0;
  }
}

bool plan_graph_step(Plan& plan, const StepArgs& a, bool with_decode, bool with_prefill,
                     void* workspace, size_t workspace_bytes) {
  plan.workspace = workspace;
  plan.workspace_bytes = workspace_bytes;
  plan.fast_decode = false;
  plan.fast_prefill = false;
  plan.n_prefill_launches = 0;
  plan.portable_mode = -1;
  plan.has_combine = false;
  plan.fused_scatter = false;
  plan.concurrent = false;
  if (a.dtype != CB_BF16) return false;
  const int G = a.num_q_heads / a.num_kv_heads;
  const int HB = std::min(a.num_kv_heads, kDecodeMaxHeads);
  const bool tile_pages_ok =
      a.block_size % 8 == 0 && (128 % a.block_size == 0 || a.block_size % 128 == 0);
  if (!((a.block_size % 16 == 0 || a.block_size == 8) && G <= 16 && a.num_kv_heads % HB == 0))
    return false;
  if (!(tile_pages_ok && G <= 16 && kRowsPerTile % G == 0)) return false;

  DecodeArgs& d = plan.decode;
  d.a = a;
  d.heads_per_cta = HB;
  d.total_units = 0;  // summed by the kernel
  d.units_on_device = 1;
  d.num_ctas = std::min(sm_count(), kMaxDecodeCtas);
  d.stage_bytes = 2 * (a.head_dim / 64) * HB * 16 * 128;
  d.q_slot_bytes = HB * G * a.head_dim * 2;
  const size_t fixed = decode_smem_bytes(0, d.stage_bytes, d.q_slot_bytes);
  d.stages = (int)std::min<size_t>(kDecodeMaxStages, (kDecodeSmemLimit - fixed) / d.stage_bytes);
  d.metadata_ready = 0;
  d.fuse_scatter = 0;
  d.k_new = d.v_new = nullptr;
  d.slot_mapping = nullptr;
  d.has_table = 0;
  const WorkspaceLayout w = layout_of(workspace_bytes, a);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  d.part_ml = reinterpret_cast<float2*>(ws + w.part_ml);
  d.part_o = reinterpret_cast<float*>(ws + w.part_o);
  plan.decode_plan.smem_bytes = decode_smem_bytes(d.stages, d.stage_bytes, d.q_slot_bytes);
  if (d.stages < 2) return false;
  plan.fast_decode = with_decode;
  combine_common(plan.combine, a, d);
  plan.combine.n_entries = -1;  // the batch's split requests are found on the device
  plan.combine.kv_per_cta = combine_kv_per_cta(a, a.num_requests);
  plan.combine.parts = 1;
  plan.has_combine = with_decode;

  PrefillArgs& pa = plan.prefill[0];
  pa.a = a;
  pa.tile_tokens = kRowsPerTile / G;
  pa.box_keys = std::min(a.block_size, 128);
  pa.n_entries = 0;
  pa.metadata_ready = 0;
  pa.k_new = pa.v_new = nullptr;  // the captured scatter launch writes the rows first
  pa.slot_mapping = nullptr;
  pa.concurrent = 0;
  pa.exit_counter = nullptr;
  pa.unit_counter = nullptr;
  pa.scatter_counter = nullptr;
  pa.device_work = 1;
  pa.total_ctas = prefill_ctas_bound(a.num_tokens, a.num_requests, pa.tile_tokens,
                                     a.num_kv_heads);
  pa.total_units = pa.total_ctas;
  pa.grid = pa.total_ctas;  // one unit per CTA, found on the device
  plan.n_prefill_launches = with_prefill ? 1 : 0;
  plan.fast_prefill = with_prefill;
  return true;
}

cudaError_t prepare_plan(const Plan& plan, const StepArgs& a) {
  cudaError_t e = cudaSuccess;
  if (plan.fast_decode) e = prepare_decode(plan.decode);
  if (e == cudaSuccess && plan.fast_prefill) e = prepare_prefill(a.head_dim);
  return e;
}

size_t workspace_extent(const Plan& plan, const StepArgs& a) {
  if (!plan.fast_decode) return kWorkspaceHeaderBytes;
  const WorkspaceLayout w = layout_of(plan.workspace_bytes, a);
  const size_t slots = (size_t)a.num_requests + (size_t)plan.decode.num_ctas;
  return w.part_o + slots * a.num_q_heads * (size_t)a.head_dim * 4;
}

size_t workspace_zeroed_prefix(const StepArgs& a, size_t workspace_bytes) {
  (void)a;
  (void)workspace_bytes;
  return kWorkspaceHeaderBytes;  // the error word and the prefill exit counter
}

cudaError_t run_plan(const Plan& plan, const StepArgs& a, cudaStream_t stream) {
  if (plan.concurrent) {
    // decode grid, the prefill grid beside it, then the merge of the split requests
    cudaError_t e = launch_decode(plan.decode, plan.decode_plan, stream);
    if (e == cudaSuccess) e = launch_prefill(plan.prefill[0], stream);
    if (e == cudaSuccess && plan.has_combine) e = launch_decode_combine(plan.combine, stream);
    return e;
  }
  if (plan.fast_decode) {
    cudaError_t e = launch_decode(plan.decode, plan.decode_plan, stream);
    if (e == cudaSuccess && plan.has_combine) e = launch_decode_combine(plan.combine, stream);
    if (e != cudaSuccess) return e;
  }
  for (int l = 0; l < plan.n_prefill_launches && plan.fast_prefill; ++l) {
    cudaError_t e = launch_prefill(plan.prefill[l], stream);
    if (e != cudaSuccess) return e;
  }
  if (plan.portable_mode >= 0) {
    cudaError_t e = launch_portable_attention(a, plan.portable_mode, stream);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace cb
