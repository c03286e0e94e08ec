// usermod.h - the run-time-compiled score_mod kernels, for the C-ABI layer.
#pragma once

#include "../../include/attn.h"

namespace attn {

// The forward, dK/dV and dQ kernels of `mod` on the current device (loaded on
// first use), as launchable pointers; ATTN_ERR_UNSUPPORTED if `mod` was built
// for the other 16-bit type.
attn_status user_mod_kernels(attn_user_mod mod, attn_dtype dtype, const void* (&kern)[3]);

// Whether `mod` was built with a mask expression (attn_user_mod_create_masked).
bool user_mod_has_mask(attn_user_mod mod);

}  // namespace attn
