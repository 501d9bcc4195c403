// attn_common.h -- host-side pieces shared by the attention block and the
// MLA decode kernel.
#pragma once

namespace tsg {
namespace attn {

// Device address of the library's attention status word on device `dev`
// (which must be current): the word a kernel reports a timeout into when
// the caller passes no status pointer, read and cleared by tsattn_status().
// Null when the lookup fails.
int* library_status_word(int dev);

}  // namespace attn
}  // namespace tsg
