// Tensor-core (tcgen05/TMEM) split-K partial kernel -- under construction.
#include "mtv_internal.cuh"

namespace mtv {

extern const int kTcRowTile = 128;
extern const int kTcKeyTile = 64;

int choose_nsplit_tc(int num_sms, int64_t pairs_per_split, int64_t max_keys, int64_t rows_total) {
  (void)rows_total;
  if (pairs_per_split <= 0) return 1;
  int64_t pairs = num_sms / 2;
  int64_t want = (pairs + pairs_per_split - 1) / pairs_per_split;
  int64_t cap = (max_keys + 255) / 256;
  if (want > cap) want = cap;
  return int(want < 1 ? 1 : want);
}

cudaError_t prepare_partial_tc() { return cudaSuccess; }

cudaError_t launch_partial_tc(const Params& P, cudaStream_t st) {
  (void)P; (void)st;
  return cudaErrorNotSupported;
}

}  // namespace mtv
