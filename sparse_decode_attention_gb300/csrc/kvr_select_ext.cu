// kvr_select_ext.cu -- the selection kernels with the optional modes
// (reranker records, magnitude-aware votes) compiled in, built as a separate
// translation unit of kvr_select.cu so both sets of instantiations compile in
// parallel.
#define KVR_SELECT_EXT_TU 1
#include "kvr_select.cu"
