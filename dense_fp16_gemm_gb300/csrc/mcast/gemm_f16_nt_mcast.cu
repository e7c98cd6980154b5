// libgemm_f16_nt_mcast.so: the GEMM library with one more kernel configuration,
// a cluster of two CTA pairs whose A rows are shared by TMA multicast
// (cluster_pairs = 2).  Same C ABI and behaviour as libgemm_f16_nt.so
// otherwise.  Built only on request, for single-GPU processes: the multicast
// configuration is taken only when the process sees exactly one GPU and A and
// B are device memory of the current device (see check_local_operands); a
// call that would need it and fails either check returns GEMM_ERR_NOT_LOCAL
// before anything is enqueued.
#define G16_MCAST_LIB 1
#include "tma_multicast.cuh"
#include "../gemm_f16_nt.cu"
