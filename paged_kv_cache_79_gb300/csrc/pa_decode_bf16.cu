// Paged decode attention: bf16 instantiations of the partition and merge kernels.
#include "pa_decode.cuh"

namespace pagedkv {

cudaError_t launch_decode_bf16(const DecodeLaunch &L, cudaStream_t stream)
{
    return launch_decode_dispatch<__nv_bfloat16>(L, stream);
}

int plan_grid_bf16(const DecodeLaunch &L) { return plan_grid_dispatch<__nv_bfloat16>(L); }

size_t decode_smem_bytes_bf16(int head_dim, int block_size, int group)
{
    return smem_dispatch<__nv_bfloat16>(head_dim, block_size, group);
}

}  // namespace pagedkv

PA_TRACE_DEFINE_READER(bf16)
