// error_words.h -- codes the kernels record in a device error word, and how
// fa_check_device turns the words it reads back into one fa_status.  Plain
// C++ (no CUDA), so a host-only test can compile it on its own.
#pragma once

#include "fa.h"  // include/fa.h (fa_status codes)

namespace fa {

// Bits a kernel ORs into its error word.
enum : unsigned int {
    kErrTimeout = 1u,    // a bounded wait ran out; the kernel unwound and its outputs are wrong
    kErrSmemAlign = 2u,  // dynamic shared memory was not 1024-byte aligned; the kernel did nothing
};

// Status for the error words of one check: `ws_word` is the word of the stream's
// workspace (fa_bwd, fa_fwd, fa_selftest_timeout), `na_word` the word of the
// no-allocation scratch (fa_bwd_noalloc).  A timeout in either wins, since it is
// the one the caller can act on (retry); any other bit is an internal error.
inline int status_from_error_words(unsigned int ws_word, unsigned int na_word) {
    const unsigned int w = ws_word | na_word;
    if (w == 0u) return FA_OK;
    if (w & kErrTimeout) return FA_ERR_TIMEOUT;
    return FA_ERR_CUDA;
}

}  // namespace fa
