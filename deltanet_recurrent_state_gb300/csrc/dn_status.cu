// dn_status_string: static descriptions of the status codes of include/dn.h.
#include "dn.h"

extern "C" const char *dn_status_string(dn_status s) {
    switch (s) {
        case DN_OK: return "DN_OK: success";
        case DN_ERR_INVALID_ARG: return "DN_ERR_INVALID_ARG: malformed argument, nothing enqueued";
        case DN_ERR_UNSUPPORTED: return "DN_ERR_UNSUPPORTED: unsupported shape or dtype, nothing enqueued";
        case DN_ERR_CUDA: return "DN_ERR_CUDA: a CUDA launch failed";
    }
    return "unknown dn_status";
}
