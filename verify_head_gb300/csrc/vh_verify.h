// Internal: the tcgen05 verify contraction serving the bf16 draft head for
// many hidden rows (not part of the public interface).
#pragma once
#include "vh_kernels.h"

namespace vh {

// Hidden rows per launch group of the bf16 draft head for a batch of B rows:
// the whole batch (up to kMaxDraftB rows) in one tcgen05 pass when B > 16 and
// H % 64 == 0, else draft_group(H).
inline int draft_launch_rows(int H, int B) { return (B > 16 && H % 64 == 0) ? kMaxDraftB : draft_group(H); }

// The verify contraction as a draft head: ids[r] = cand[winning row] and
// maxlogit[r] its score for nb <= 256 hidden rows of width H % 64 == 0 over
// the n_rows-row table W; no acceptance scan.  With cand ascending (the draft
// head's precondition) the lowest row on ties is the lowest id.
cudaError_t launch_draft_tc(const uint16_t* x, int nb, int H, const uint16_t* W, const int32_t* cand, int n_rows,
                            Workspace ws, int32_t* ids, float* maxlogit, cudaStream_t s);

}  // namespace vh
