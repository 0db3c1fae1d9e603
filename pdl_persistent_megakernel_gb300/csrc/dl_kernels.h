// dl_kernels.h -- host-visible entry points of dl_kernels.cu.
#pragma once

#include <cuda_runtime.h>

#include "dl_internal.h"

namespace dl {

const void* gemm_kernel(int mma, int m_or_mp);
// The add + RMSNorm kernel for rows of H columns, each row split over a
// cluster of `split` CTAs (1, 2 or 4); NULL for an unsupported pair.
const void* norm_kernel(int H, int split);
const void* attn_kernel(int QRp);
const void* attn_tc_kernel();
int attn_tc_smem_bytes(int QRp, int stages);
const void* mega_kernel();
cudaError_t launch_bind(Binding* dst, const Binding& v, cudaStream_t s);
int gemm_smem_bytes(int npair, int Mp, int stages, int KB, int fp8, int epi, int M, int share);
int attn_smem_bytes(int QRp, int stages);
// CTAs of a split-KV attention over `pairs` (request, kv head) streams of
// `nb` 64-key blocks on `sms` SMs (dl_host.cu).
int attn_ctas(int pairs, int nb, int sms, int min_blocks = 1);
// Pipeline stages of the mma.sync attention kernel for a query-row padding
// (dl_host.cu): one rule for the plans and the allocation-free entry point,
// so the kernel's shared-memory attribute is the same whichever sets it.
int attn_mma_stages(int QRp);
int norm_smem_bytes();
cudaError_t launch_test_kv_write(const void* src, void* kv, const int* bt, const int* pos,
                                 int layer, int M, int T, int Hkv, int d, int P,
                                 int num_pages, int max_pages, DevStatus* st,
                                 cudaStream_t s);
cudaError_t launch_test_kv_gather(const void* kv, const int* bt, void* dst, int layer, int R,
                                  int n_keys, int Hkv, int d, int P, int num_pages,
                                  int max_pages, DevStatus* st, cudaStream_t s);

}  // namespace dl
