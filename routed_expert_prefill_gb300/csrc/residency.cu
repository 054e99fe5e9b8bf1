// Residency plan of the streamed routed records, and the streaming context.
//
// The rules (cherenkov qwen4_exp engine, prefill/experts.rs,
// prepare_expert_jobs and pf_experts; prefill.rs RING / GROUP): the experts
// with rows are ranked by row count and the first pool_slots stay resident;
// the others stream through a ring of slots; the copies go in fetch batches
// and a batch overwrites ring slots only once the batch that last read them
// has finished.  Where the pages leave the pool's eviction open, a kept
// expert takes the lowest free slot, else the least recently used slot whose
// expert has no rows in this chunk.
#include <algorithm>
#include <cstring>

#include "common.cuh"
#include "residency.cuh"

namespace moe {

int plan_residency(const int32_t* counts, int E, const moe_stream_cfg& cfg, int64_t call, moe_residency_plan& pl) {
  const int P = cfg.pool_slots, R = cfg.ring_slots, G = cfg.group;
  // experts by row count, descending, ties to the lower id
  std::vector<int32_t> order;
  order.reserve(E);
  for (int e = 0; e < E; ++e)
    if (counts[e] > 0) order.push_back(e);
  std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return counts[a] > counts[b]; });

  // slot of each resident expert; the pool table must name distinct experts
  std::vector<int32_t> slot_of(E, -1);
  for (int s = 0; s < P; ++s) {
    const int e = pl.pool_expert[s];
    if (e < -1 || e >= E) return set_error(MOE_EINVAL, "pool slot %d holds expert %d, outside [-1, %d)", s, e, E);
    if (e < 0) continue;
    if (slot_of[e] >= 0) return set_error(MOE_EINVAL, "expert %d is in pool slots %d and %d", e, slot_of[e], s);
    slot_of[e] = s;
  }
  // free slots ascending; evictable slots (resident expert without rows
  // now) by last use, then slot.  Neither list changes while the keep set
  // is placed: a slot taken from either then holds an expert with rows.
  std::vector<int32_t> free_s, victims;
  for (int s = 0; s < P; ++s) {
    const int e = pl.pool_expert[s];
    if (e < 0)
      free_s.push_back(s);
    else if (counts[e] <= 0)
      victims.push_back(s);
  }
  std::sort(victims.begin(), victims.end(), [&](int a, int b) {
    return pl.pool_last[a] != pl.pool_last[b] ? pl.pool_last[a] < pl.pool_last[b] : a < b;
  });
  std::vector<uint8_t> fill(E, 0);
  size_t fi = 0, vi = 0;
  const int n_keep = std::min<int>(P, (int)order.size());
  for (int i = 0; i < n_keep; ++i) {
    const int e = order[i];
    if (slot_of[e] >= 0) continue;
    int s;
    if (fi < free_s.size()) {
      s = free_s[fi++];
    } else if (vi < victims.size()) {
      s = victims[vi++];
      slot_of[pl.pool_expert[s]] = -1;
    } else {
      continue;  // no room: streams for this chunk
    }
    pl.pool_expert[s] = e;
    slot_of[e] = s;
    fill[e] = 1;
  }

  // jobs in ascending expert order
  int nc = 0, ring_pos = 0;
  for (int e = 0; e < E; ++e) {
    if (counts[e] <= 0) {
      pl.rec[e] = -1;
      pl.batch[e] = -1;
      continue;
    }
    int slot;
    bool copy;
    if (slot_of[e] >= 0) {
      slot = slot_of[e];
      pl.pool_last[slot] = call;
      copy = fill[e] != 0;
    } else {
      slot = P + ring_pos % R;
      ++ring_pos;
      copy = true;
    }
    pl.rec[e] = slot;
    if (copy) {
      pl.copy_expert[nc] = e;
      pl.copy_slot[nc] = slot;
      pl.batch[e] = 1 + nc / G;
      ++nc;
    } else {
      pl.batch[e] = 0;
    }
  }
  pl.n_copies = nc;
  pl.n_batches = 1 + (nc + G - 1) / G;
  const int lag = R / G;
  pl.wait_for[0] = 0;
  for (int b = 1; b < pl.n_batches; ++b) pl.wait_for[b] = b - lag >= 1 ? b - lag : 0;
  return MOE_OK;
}

}  // namespace moe

using namespace moe;

namespace {

int check_cfg(const moe_stream_cfg* cfg) {
  if (!cfg) return set_error(MOE_EINVAL, "cfg is NULL");
  if (cfg->pool_slots < 0) return set_error(MOE_EINVAL, "pool_slots=%d is negative", cfg->pool_slots);
  if (cfg->group < 1) return set_error(MOE_EINVAL, "group=%d must be at least 1", cfg->group);
  if (cfg->ring_slots < cfg->group || cfg->ring_slots % cfg->group)
    return set_error(MOE_EINVAL, "ring_slots=%d must be a positive multiple of group=%d", cfg->ring_slots,
                     cfg->group);
  const int mb = cfg->miss_bits;
  if (mb != 0 && mb != 2 && mb != 3 && mb != 4 && mb != 8)
    return set_error(MOE_EINVAL, "miss_bits=%d: 0, 2, 3, 4 or 8", mb);
  return MOE_OK;
}

// Record bytes at the pool's and at the ring's code width (0 on bad dims).
void record_sizes(const moe_dims* dims, const moe_stream_cfg* cfg, size_t& base, size_t& miss, int& miss_bits) {
  base = moe_packed_bytes(dims, 0) / dims->E;
  moe_dims dm = *dims;
  miss_bits = cfg->miss_bits ? cfg->miss_bits : (dims->bits ? dims->bits : 4);
  dm.bits = miss_bits;
  miss = moe_packed_bytes(&dm, 0) / dims->E;
}

}  // namespace

extern "C" {

int moe_plan_residency(const int32_t* counts, int32_t E, const moe_stream_cfg* cfg, int64_t call,
                       moe_residency_plan* plan) {
  int s;
  if ((s = check_cfg(cfg)) != MOE_OK) return s;
  if (E < 1 || E > 1024) return set_error(MOE_ESHAPE, "E=%d outside [1, 1024]", E);
  if (!counts || !plan) return set_error(MOE_EINVAL, "counts or plan is NULL");
  if (!plan->rec || !plan->batch || !plan->copy_expert || !plan->copy_slot || !plan->wait_for ||
      (cfg->pool_slots > 0 && (!plan->pool_expert || !plan->pool_last)))
    return set_error(MOE_EINVAL, "a plan array is NULL");
  return plan_residency(counts, E, *cfg, call, *plan);
}

size_t moe_stream_slot_bytes(const moe_dims* dims, const moe_stream_cfg* cfg) {
  if (!dims || dims->E < 1 || dims->E > 1024 || check_cfg(cfg) != MOE_OK) return 0;
  size_t rec, miss;
  int miss_bits;
  record_sizes(dims, cfg, rec, miss, miss_bits);
  if (rec == 0 || miss == 0) return 0;
  return (size_t)cfg->pool_slots * rec + (size_t)cfg->ring_slots * miss;
}

int moe_streamer_create(const moe_dims* dims, const moe_stream_cfg* cfg, moe_streamer** out) {
  if (!out) return set_error(MOE_EINVAL, "out is NULL");
  *out = nullptr;
  if (!dims) return set_error(MOE_EINVAL, "dims is NULL");
  if (dims->E < 1 || dims->E > 1024) return set_error(MOE_ESHAPE, "E=%d outside [1, 1024]", dims->E);
  int s;
  if ((s = check_cfg(cfg)) != MOE_OK) return s;
  size_t rec, miss;
  int miss_bits;
  record_sizes(dims, cfg, rec, miss, miss_bits);  // 0 on bad dims, message set
  if (rec == 0 || miss == 0) return MOE_ESHAPE;
  moe_streamer* st = new moe_streamer();
  st->dims = *dims;
  st->cfg = *cfg;
  st->rec_bytes = rec;
  st->miss_bits = miss_bits;
  st->miss_bytes = miss;
  st->call = 0;
  const int E = dims->E, P = cfg->pool_slots;
  st->pool_expert.assign(P, -1);
  st->pool_last.assign(P, 0);
  st->counts.assign(E, 0);
  st->copy_expert.assign(E, 0);
  st->copy_slot.assign(E, 0);
  st->wait_for.assign(E + 1, 0);
  st->plan_rec.assign(E, -1);
  st->plan_batch.assign(E, -1);
  auto fail = [&](cudaError_t e, const char* what) {
    moe_streamer_destroy(st);
    return set_error(MOE_ECUDA, "moe_streamer_create: %s: %s", what, cudaGetErrorString(e));
  };
  cudaError_t e;
  if ((e = cudaGetDevice(&st->device)) != cudaSuccess) return fail(e, "cudaGetDevice");
  if ((e = cudaHostAlloc(&st->h_offsets, (E + 1) * sizeof(int32_t), cudaHostAllocDefault)) != cudaSuccess)
    return fail(e, "cudaHostAlloc");
  if ((e = cudaHostAlloc(&st->h_maps, (2 * E + 1) * sizeof(int32_t), cudaHostAllocDefault)) != cudaSuccess)
    return fail(e, "cudaHostAlloc");
  if ((e = cudaMalloc(&st->d_maps, (2 * E + 1) * sizeof(int32_t))) != cudaSuccess) return fail(e, "cudaMalloc");
  if ((e = cudaStreamCreateWithFlags(&st->copy, cudaStreamNonBlocking)) != cudaSuccess)
    return fail(e, "cudaStreamCreate");
  if ((e = cudaEventCreateWithFlags(&st->fetched, cudaEventDisableTiming)) != cudaSuccess)
    return fail(e, "cudaEventCreate");
  if ((e = cudaEventCreateWithFlags(&st->call_done, cudaEventDisableTiming)) != cudaSuccess)
    return fail(e, "cudaEventCreate");
  st->done.assign(cfg->ring_slots / cfg->group, nullptr);
  for (auto& ev : st->done)
    if ((e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming)) != cudaSuccess) return fail(e, "cudaEventCreate");
  *out = st;
  return MOE_OK;
}

int moe_streamer_destroy(moe_streamer* st) {
  if (!st) return MOE_OK;
  // kernels of earlier calls may still read the device maps, and copies
  // the pinned staging: let the device finish first
  cudaDeviceSynchronize();
  for (auto ev : st->done)
    if (ev) cudaEventDestroy(ev);
  if (st->fetched) cudaEventDestroy(st->fetched);
  if (st->call_done) cudaEventDestroy(st->call_done);
  if (st->copy) cudaStreamDestroy(st->copy);
  if (st->d_maps) cudaFree(st->d_maps);
  if (st->h_maps) cudaFreeHost(st->h_maps);
  if (st->h_offsets) cudaFreeHost(st->h_offsets);
  delete st;
  return MOE_OK;
}

int moe_streamer_pool(const moe_streamer* st, int32_t* pool_expert, int32_t n) {
  if (!st || (!pool_expert && n > 0)) return set_error(MOE_EINVAL, "streamer or pool_expert is NULL");
  const int m = std::min<int>(n, st->cfg.pool_slots);
  if (m > 0) std::memcpy(pool_expert, st->pool_expert.data(), m * sizeof(int32_t));
  return m;
}

}  // extern "C"
