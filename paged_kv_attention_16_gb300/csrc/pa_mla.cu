// pa_mla.cu -- absorbed-MLA decode.
#include "pa_internal.h"

extern "C" {

size_t pa_mla_decode_workspace_bytes(int, int, int, int, int) { return 0; }

pa_status pa_mla_decode(const void *, const void *, const int32_t *, const int32_t *, int, int,
                        int, int, float, void *, void *, int, int, int, int, int) {
  return PA_ERR_UNSUPPORTED;
}

}  // extern "C"
