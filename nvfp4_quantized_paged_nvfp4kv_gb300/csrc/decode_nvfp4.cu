// NVFP4 paged decode: instantiation and launcher.
#include "decode_common.cuh"

namespace nvfp4kv {

template <class Fmt, bool kMulti>
static cudaError_t launch_decode(const DecodeParams &p, cudaStream_t s)
{
    const size_t smem = decode_smem_bytes<Fmt>(p.batch);
    cudaError_t e = cudaFuncSetAttribute(decode_kernel<Fmt, kMulti>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess)
        return e;
    const int grid = (p.num_workers + kDecodeWarps - 1) / kDecodeWarps;
    return launch_pdl(decode_kernel<Fmt, kMulti>, dim3(grid), dim3(kDecodeWarps * 32), smem, s, p);
}

cudaError_t launch_decode_nvfp4(const DecodeParams &p, cudaStream_t s)
{
    return launch_decode<Nvfp4Format, false>(p, s);
}

cudaError_t launch_decode_nvfp4_multi(const DecodeParams &p, cudaStream_t s)
{
    return launch_decode<Nvfp4Format, true>(p, s);
}

} // namespace nvfp4kv
