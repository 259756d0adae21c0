// Shape dispatch and the per-path launch sequences.
#pragma once

#include <cuda_runtime.h>

#include "internal.h"

namespace tl {

// Extra device bytes create() packs after the plain parameters (re-laid-out
// weights some paths want), and the routine that fills them.
size_t packed_extra_bytes(const tl_encoder* h);
cudaError_t pack_extra(tl_encoder* h, void* dst, size_t bytes);

// The path forward() runs: the forced one if it can run the shape, the
// frozen shape table's choice under TL_PATH_AUTO; TL_PATH_AUTO itself means
// "no path can run this shape".
tl_path choose_path(const tl_encoder* h, int B, int L);
// The split-K attention setting forward() uses for B x L: the handle's own
// (tl_encoder_set_attention_split) unless it is automatic, then the frozen
// table's entry for the shape if there is one, else automatic (-1).
int attention_split_setting(const tl_encoder* h, int B, int L);
size_t path_workspace_bytes(const tl_encoder* h, tl_path p, int B, int L);
cudaError_t run_path(tl_encoder* h, tl_path p, const void* x, int B, int L,
                     const int32_t* valid_len, void* out, void* ws, cudaStream_t s);

}  // namespace tl
