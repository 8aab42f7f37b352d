// The packed-sequence (varlen) instances of the attention backward.
#define ATTN_BWD_INST_VARLEN true
#include "attn_bwd_inst.cu"
