// kvr_select_att.cu -- the selection kernels with the fused attention tail
// (selection + attention of a decode step in one cluster launch), built as a
// separate translation unit of kvr_select.cu so the instantiations compile in
// parallel with the others.
#define KVR_SELECT_ATT_TU 1
#include "kvr_select.cu"
