// eg_tuning.cu -- dispatch: token-bucket lookup in the swept tuning table,
// then a default rule.  The pages tune each decode shape on its own at
// num_tokens in {1, 2, 4, 8, 16, 24, 32} ("Helion linear backend in vLLM",
// sections "Hybrid dispatch" and "How the autotuner searches"), and ship a
// default configuration for functional tests next to the tuned sets
// (section "How it will be deployed").  Above 32 tokens the pages hand the
// layer to library kernels; here the same kernel keeps going, with swept
// entries at 64, 128, ..., 2048 tokens (a token count uses the first bucket
// at or above it).
#include "eg_registry.h"
#include "eg_tuning.h"

namespace eg {

namespace {

// Rows written by the offline sweep (bench/sweep tool); empty until swept.
const TuningRow kTable[] = {
#include "eg_tuning_table.inc"
    {-1, -1, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0}};

// decode buckets, then the mid-range (prefill ramp) buckets
constexpr int kBuckets[] = {1, 2, 4, 8, 16, 24, 32, 64, 128, 256, 512, 1024, 2048};

int bucket_of(int64_t M) {
  for (int b : kBuckets)
    if (M <= b) return b;
  return 0;
}

bool entry_for(const eg_problem& p, int swap, int bn, KernelEntry* ke) {
  if (p.flags & EG_EPI_GATED) {
    if (p.dtype == EG_IN_BF16) return lookup_bf16_gated(swap, bn, ke);
    if (p.dtype == EG_IN_E4M3 && p.scale == EG_SCALE_TOKEN_CHANNEL)
      return lookup_e4m3_tc_gated(swap, bn, ke);
    return false;
  }
  if (p.dtype == EG_IN_BF16) return lookup_bf16(swap, bn, ke);
  if (p.dtype == EG_IN_E4M3 && p.scale == EG_SCALE_TOKEN_CHANNEL) return lookup_e4m3_tc(swap, bn, ke);
  if (p.dtype == EG_IN_E4M3 && p.scale == EG_SCALE_BLOCK) return lookup_e4m3_block(swap, bn, ke);
  if (p.dtype == EG_IN_INT8) return lookup_int8_tc(swap, bn, ke);
  return false;
}

constexpr uint32_t kSmemPerSm = 233472;  // shared memory per SM on sm_100/103
constexpr uint32_t kSmemPerBlock = 232448;

}  // namespace

bool tuning_default(const eg_problem& p, int sms, eg_tuning* out) {
  const bool promote = p.scale == EG_SCALE_BLOCK || p.dtype == EG_IN_INT8;
  eg_tuning t{};
  if (p.M <= 64) {
    // decode: rows over N (swap-AB), columns over the few tokens
    t.swap_ab = 1;
    t.tile_n = p.M <= 16 ? 16 : (p.M <= 32 ? 32 : 64);
    // INT8: a deep int8 staging ring (the fp16 operand ring is separate)
    t.stages = (p.dtype == EG_IN_INT8) ? 8 : 4;
  } else {
    t.swap_ab = 0;
    const bool gated = (p.flags & EG_EPI_GATED) != 0;  // tiles 64 and 128 (two accumulators)
    const int max_bn = (p.dtype == EG_IN_INT8 || (gated && p.N <= 64)) ? 64
                       : (promote || gated) ? 128 : 256;
    int bn = gated ? 64 : 16;
    while (bn < max_bn && bn < p.N) bn *= 2;
    t.tile_n = bn;
    t.stages = 8;
  }
  KernelEntry ke;
  if (!entry_for(p, t.swap_ab, t.tile_n, &ke)) return false;
  const uint32_t extra = static_cast<uint32_t>(
      block_scale_smem_bytes(p, t.swap_ab, t.tile_n, ke.elems_per_stage));
  while (t.stages > 2 && ke.fixed_bytes + uint32_t(t.stages) * ke.stage_bytes + extra > kSmemPerBlock)
    --t.stages;
  const uint32_t smem = ke.fixed_bytes + uint32_t(t.stages) * ke.stage_bytes + extra;
  int per_sm = static_cast<int>(kSmemPerSm / (smem + 1024));
  if (per_sm < 1) per_sm = 1;
  if (per_sm > 2) per_sm = 2;
  const int64_t rows = t.swap_ab ? p.N : p.M, cols = t.swap_ab ? p.M : p.N;
  const int64_t tiles = ((rows + 127) / 128) * ((cols + t.tile_n - 1) / t.tile_n);
  const int64_t k_tiles = (p.K + ke.elems_per_stage - 1) / ke.elems_per_stage;
  int64_t split = 1;
  if (tiles > 0 && tiles < sms) split = (int64_t(sms) * per_sm) / tiles;
  if (split > k_tiles / 2) split = k_tiles / 2;  // keep >= 2 K tiles per split
  if (split > 256) split = 256;
  if (split < 1) split = 1;
  t.split_k = static_cast<int32_t>(split);
  *out = t;
  return true;
}

int32_t epi_class_of(const eg_problem& p) {
  if (p.flags & EG_EPI_GATED) return EPI_CLASS_GATED;
  if (p.flags & EG_RUN_QUANT_A) return EPI_CLASS_QUANT;
  return EPI_CLASS_PLAIN;
}

namespace {

const TuningRow* find_row(const eg_problem& p, int bucket, int32_t epi) {
  for (const TuningRow& r : kTable) {
    if (r.dtype < 0) break;
    if (r.dtype == p.dtype && r.scale == p.scale && r.N == p.N && r.K == p.K && r.m_max == bucket &&
        r.epi == epi)
      return &r;
  }
  return nullptr;
}

}  // namespace

bool tuning_lookup(const eg_problem& p, int sms, eg_tuning* out) {
  // rows of the problem's own epilogue class first; the quantisation
  // prologue's GEMM is the plain layer's, so it falls back to the plain
  // rows; a gated unit (twice the weights, two accumulators) to the rule
  const int b = bucket_of(p.M);
  const int32_t epi = epi_class_of(p);
  const TuningRow* r = find_row(p, b, epi);
  if (!r && epi == EPI_CLASS_QUANT) r = find_row(p, b, EPI_CLASS_PLAIN);
  if (r) {
    *out = eg_tuning{r->tile_n, r->stages, r->split_k, r->swap_ab, r->stream_k, r->cluster_reduce,
                     r->cta_pair};
    return true;
  }
  return tuning_default(p, sms, out);
}

}  // namespace eg
