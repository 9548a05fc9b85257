// Attention entry points (forward / backward kernels follow).
#include "lpfa_internal.h"

extern "C" size_t lpfa_fwd_workspace_size(const lpfa_attn_desc* desc) {
  (void)desc;
  return 256;
}
extern "C" size_t lpfa_bwd_workspace_size(const lpfa_attn_desc* desc) {
  (void)desc;
  return 256;
}
extern "C" lpfa_status lpfa_fwd(const lpfa_attn_desc*, const void*, const void*,
                                const void*, const void*, const void*,
                                const void*, void*, float*, void*, size_t,
                                void*) {
  return LPFA_ERR_UNSUPPORTED;
}
extern "C" lpfa_status lpfa_bwd(const lpfa_attn_desc*, const void*, const void*,
                                const void*, const void*, const void*,
                                const void*, const void*, const void*,
                                const void*, const void*, const void*,
                                const void*, const void*, const float*, void*,
                                void*, void*, void*, size_t, void*) {
  return LPFA_ERR_UNSUPPORTED;
}
