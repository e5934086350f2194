// Host-only: the block-aligned split of a tensor list over the processes of a
// ZeRO-style sharded optimizer step.
//
// "Яндекс Публикует ЯЛМ 100Б" (Yandex's YaLM-100B training notes), section
// "ZeRO" under "Случай с несколькими графическими процессорами": every
// process is given one group of the parameters, keeps their values and
// optimizer state, and is the only one to update them, so the optimizer step
// costs O(N / P) per process; the gradients are reduced before the step and
// the parameters gathered by every process after it.  Blocks of 2048
// elements are normalised independently ("8-BIT OPTIMIZERS VIA BLOCK-WISE
// QUANTIZATION", section 二 / 逐块量化), so cutting on block boundaries keeps
// every block, and with it the sharded step, identical to the unsharded one.
//
// Layout: tensor i occupies blocks [B_i, B_i + ceil(n_i / 2048)) of a padded
// flat space (B the prefix sums of the block counts, NB their total); rank r
// owns the K = ceil(NB / P) blocks [r K, (r + 1) K) clipped to NB.  Equal
// shares let the collectives move equal-sized slices of the padded buffers.
#include <cstdint>

#include "bwd.h"
#include "host_util.h"

using bwd::host::fail;

extern "C" bwd_status bwd_zero_shard(int32_t num_tensors, const int64_t* n, int32_t world, int32_t rank,
                                     int64_t* blocks_per_rank, int32_t* num_pieces, int32_t* tensor,
                                     int64_t* offset, int64_t* count) {
  if (num_tensors < 0) return fail(BWD_ERR_INVALID_ARG, "num_tensors < 0");
  if (world < 1 || rank < 0 || rank >= world)
    return fail(BWD_ERR_INVALID_ARG, "need 1 <= world and 0 <= rank < world (got %d, %d)", world, rank);
  if (!num_pieces || (num_tensors > 0 && !n)) return fail(BWD_ERR_INVALID_ARG, "NULL pointer");
  int64_t nb_total = 0;
  for (int32_t i = 0; i < num_tensors; ++i) {
    if (n[i] < 0) return fail(BWD_ERR_INVALID_ARG, "tensor %d: n < 0", i);
    const int64_t nb = bwd_num_blocks(n[i]);
    if (nb_total > INT64_MAX / BWD_BLOCK - nb) return fail(BWD_ERR_INVALID_ARG, "total size overflows");
    nb_total += nb;
  }
  const int64_t k = (nb_total + world - 1) / world;
  const int64_t lo = k * rank;
  const int64_t hi = lo + k < nb_total ? lo + k : nb_total;
  if (blocks_per_rank) *blocks_per_rank = k;
  int32_t pieces = 0;
  int64_t b0 = 0;  // first block of tensor i
  for (int32_t i = 0; i < num_tensors && b0 < hi; ++i) {
    const int64_t nb = bwd_num_blocks(n[i]);
    const int64_t a = b0 > lo ? b0 : lo;
    const int64_t b = b0 + nb < hi ? b0 + nb : hi;
    if (a < b) {
      const int64_t first = (a - b0) * BWD_BLOCK;
      const int64_t end = (b - b0) * BWD_BLOCK < n[i] ? (b - b0) * BWD_BLOCK : n[i];
      if (tensor) tensor[pieces] = i;
      if (offset) offset[pieces] = first;
      if (count) count[pieces] = end - first;
      ++pieces;
    }
    b0 += nb;
  }
  *num_pieces = pieces;
  return BWD_OK;
}
