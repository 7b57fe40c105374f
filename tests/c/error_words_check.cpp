// Host-only check of how fa_check_device turns the device error words it reads
// (the stream workspace's and the no-allocation scratch's) into one status.
// Exits 0 when every case holds, else prints the failing case and exits 1.
#include <stdio.h>

#include "error_words.h"

int main() {
    using fa::status_from_error_words;
    struct Case {
        unsigned ws, na;
        int want;
    } cases[] = {
        {0u, 0u, FA_OK},
        {fa::kErrTimeout, 0u, FA_ERR_TIMEOUT},            // fa_bwd / fa_fwd timed out
        {0u, fa::kErrTimeout, FA_ERR_TIMEOUT},            // fa_bwd_noalloc timed out
        {fa::kErrTimeout, fa::kErrTimeout, FA_ERR_TIMEOUT},
        {fa::kErrSmemAlign, 0u, FA_ERR_CUDA},             // internal error, no timeout
        {0u, fa::kErrSmemAlign, FA_ERR_CUDA},
        {fa::kErrSmemAlign, fa::kErrTimeout, FA_ERR_TIMEOUT},
        {fa::kErrTimeout | fa::kErrSmemAlign, 0u, FA_ERR_TIMEOUT},
        {0x80u, 0u, FA_ERR_CUDA},                         // an unknown bit is still an error
    };
    int bad = 0;
    for (const Case& c : cases) {
        const int got = status_from_error_words(c.ws, c.na);
        if (got != c.want) {
            printf("ws=%#x na=%#x: got %d, want %d\n", c.ws, c.na, got, c.want);
            bad = 1;
        }
    }
    return bad;
}
