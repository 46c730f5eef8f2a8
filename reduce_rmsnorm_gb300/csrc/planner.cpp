// Wave-aware prefix/suffix token split (pure host integer code, no CUDA).
//
// [W] = "TokenWeave: Why Hiding Tensor-Parallel Communication Needs Wave
// Arithmetic, Not Finer Tiles". "The overlap trap": a c-CTA kernel on S SMs
// runs in ceil(c/S) waves. "Fix one: split at wave boundaries, unequally":
// split the batch exactly twice, prefix = half + offset, suffix = half -
// offset, offsets from {0, 64, 128, 192, 256, 512} below half, keeping the
// waves of the two pieces within the unsplit count; one-wave kernels and
// batches under the 1K-token threshold are not split. The worked example
// (132 / 168 of 300 CTAs) puts the smaller piece first, so offsets are tried
// with both signs, smallest |offset| first and the smaller prefix on a tie.
// "Fix one" also describes the pages' own rule, an offline timed sweep whose
// winners go in a lookup table; tw_split_lookup consults such a table and
// falls back to the wave constraint.
#include <algorithm>
#include <cstdint>
#include <vector>

#include "tw.h"

namespace {

const int64_t kDefaultOffsets[] = {0, 64, 128, 192, 256, 512};  // sorted, unique
const int kDefaultMinSplitTokens = 1024;

int64_t ceil_div(int64_t a, int64_t b) { return a / b + (a % b != 0); }  // a >= 0, b > 0

// CTAs of a t-token piece of a T-token, C-CTA kernel: ceil(t * C / T).
int64_t piece_ctas(int64_t t, int64_t T, int64_t C) {
  const __int128 n = static_cast<__int128>(t) * C;
  return static_cast<int64_t>(n / T + (n % T != 0));
}

}  // namespace

extern "C" int tw_wave_split(int64_t num_tokens, int64_t ctas_unsplit, int num_sms,
                             const tw_split_opts* opts, int64_t* prefix_tokens,
                             int64_t* suffix_tokens) {
  if (!prefix_tokens || !suffix_tokens) return TW_ERR_INVALID_ARG;
  if (num_tokens < 0 || ctas_unsplit < 0 || num_sms <= 0) return TW_ERR_INVALID_ARG;

  bool every_offset = false;
  // The default offsets are used in place; a caller's list is copied, sorted
  // and deduplicated (no exception leaves this function).
  const int64_t* offsets = kDefaultOffsets;
  size_t n_offsets = sizeof(kDefaultOffsets) / sizeof(kDefaultOffsets[0]);
  std::vector<int64_t> custom;
  int64_t min_split = kDefaultMinSplitTokens;
  if (opts) {
    if (opts->n_offsets < 0) return TW_ERR_INVALID_ARG;
    if (!opts->offsets && opts->n_offsets > 0) return TW_ERR_INVALID_ARG;
    if (!opts->offsets) {
      every_offset = true;
    } else {
      for (int i = 0; i < opts->n_offsets; ++i)
        if (opts->offsets[i] < 0) return TW_ERR_INVALID_ARG;
      try {
        custom.assign(opts->offsets, opts->offsets + opts->n_offsets);
      } catch (...) {
        return TW_ERR_INVALID_ARG;  // a list too large to copy
      }
      std::sort(custom.begin(), custom.end());
      custom.erase(std::unique(custom.begin(), custom.end()), custom.end());
      offsets = custom.data();
      n_offsets = custom.size();
    }
    min_split = opts->min_split_tokens;
  }

  const int64_t T = num_tokens, C = ctas_unsplit, S = num_sms;
  *prefix_tokens = T;
  *suffix_tokens = 0;
  if (T == 0) return TW_OK;
  const int64_t unsplit_waves = ceil_div(C, S);
  if (T < min_split || unsplit_waves <= 1) return TW_OK;

  const int64_t half = T / 2;
  auto admissible = [&](int64_t p) {
    return ceil_div(piece_ctas(p, T, C), S) + ceil_div(piece_ctas(T - p, T, C), S) <= unsplit_waves;
  };
  auto try_offset = [&](int64_t off) {
    if (admissible(half - off)) {
      *prefix_tokens = half - off;
    } else if (off > 0 && admissible(half + off)) {
      *prefix_tokens = half + off;
    } else {
      return false;
    }
    *suffix_tokens = T - *prefix_tokens;
    return true;
  };

  if (every_offset) {
    for (int64_t off = 0; off < half; ++off)
      if (try_offset(off)) return TW_OK;
    return TW_OK;
  }
  for (size_t i = 0; i < n_offsets; ++i) {
    if (offsets[i] >= half) break;
    if (try_offset(offsets[i])) return TW_OK;
  }
  return TW_OK;
}

extern "C" int tw_split_lookup(const int64_t* table_tokens, const int64_t* table_prefix,
                               int n_entries, int64_t num_tokens, int64_t ctas_unsplit,
                               int num_sms, const tw_split_opts* opts, int64_t* prefix_tokens,
                               int64_t* suffix_tokens) {
  if (!prefix_tokens || !suffix_tokens || n_entries < 0) return TW_ERR_INVALID_ARG;
  if (n_entries > 0 && (!table_tokens || !table_prefix)) return TW_ERR_INVALID_ARG;
  if (num_tokens < 0) return TW_ERR_INVALID_ARG;
  for (int i = 0; i < n_entries; ++i) {
    if (table_tokens[i] != num_tokens) continue;
    const int64_t p = table_prefix[i];
    if (p < 0 || p > num_tokens) return TW_ERR_INVALID_ARG;
    *prefix_tokens = p;
    *suffix_tokens = num_tokens - p;
    return TW_OK;
  }
  return tw_wave_split(num_tokens, ctas_unsplit, num_sms, opts, prefix_tokens, suffix_tokens);
}

// Token-boundary shard of one rank ([W] "Fix two": the reduce-scatter splits
// the batch at token boundaries, so each rank normalises whole token rows).
// Every rank's shard holds ceil(T / world) rows except at the tail: rank r
// owns [min(r * s, T), min((r + 1) * s, T)) with s = ceil(T / world), so the
// shards are contiguous, disjoint, in rank order, and cover every row once.
extern "C" int tw_shard_rows(int64_t num_tokens, int world, int rank, int64_t* row0,
                             int64_t* rows) {
  if (!row0 || !rows) return TW_ERR_INVALID_ARG;
  if (num_tokens < 0 || world <= 0 || rank < 0 || rank >= world) return TW_ERR_INVALID_ARG;
  const int64_t s = ceil_div(num_tokens, world);
  const int64_t a = std::min<int64_t>(static_cast<int64_t>(rank) * s, num_tokens);
  const int64_t b = std::min<int64_t>(a + s, num_tokens);
  *row0 = a;
  *rows = b - a;
  return TW_OK;
}
