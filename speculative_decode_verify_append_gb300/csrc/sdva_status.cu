// sdva_status.cu -- host-side descriptions of return codes and status bits.
#include "sdva.h"

extern "C" const char* sdva_status_string(int code) {
  switch (code) {
    case SDVA_OK:
      return "ok";
    case SDVA_ERR_INVALID:
      return "invalid argument (null pointer, non-positive size or q heads not a multiple of kv heads)";
    case SDVA_ERR_UNSUPPORTED:
      return "unsupported configuration (head_dim must be 128, page_size 64, window <= 16, known kv dtype)";
    case SDVA_ERR_WORKSPACE:
      return "workspace missing, misaligned or smaller than verify_attn_workspace_size()";
    case SDVA_ERR_CUDA:
      return "CUDA launch failed";
    case SDVA_STATUS_BAD_PAGE:
      return "device status: a page_table entry is outside [0, num_pages)";
    case SDVA_STATUS_OVERFLOW:
      return "device status: a lane's length does not fit its page table row or max_context";
    case SDVA_STATUS_BAD_DRAFT:
      return "device status: a draft id is outside [0, vocab)";
    case SDVA_STATUS_TIMEOUT:
      return "device status: a bounded device wait timed out";
    case SDVA_STATUS_BAD_TREE:
      return "device status: a draft tree's parent is not an earlier slot";
    case SDVA_STATUS_BAD_COUNT:
      return "device status: a per-lane draft or token count is out of range";
    default:
      return code > 0 ? "device status: several bits set" : "unknown code";
  }
}
