// tcgen05 split-KV chunk kernel: instantiations, TMA tensor maps and launch.
#include <cudaTypedefs.h>

#include <atomic>
#include <cstring>

#include "split_kv_chunk_tc.cuh"

namespace kvd {

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static std::atomic<void*> fn{nullptr};
    void* f = fn.load(std::memory_order_acquire);
    if (!f) {
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        fn.store(f, std::memory_order_release);
    }
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
}

// bf16 tensor map with 128-byte swizzle; dims/strides innermost first (strides in bytes).
bool encode(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
            const cuuint32_t* box, bool swizzle = true) {
    auto enc = encode_fn();
    if (!enc) return false;
    const cuuint32_t es[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

template <int D, bool F32>
cudaError_t launch_tc_chunk(const ChunkKernel& k, const DecodeParams& p, cudaStream_t stream) {
    TcMaps maps;
    std::memset(&maps, 0, sizeof maps);
    {
        const cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)p.B * p.Hq};
        const cuuint64_t strides[1] = {(cuuint64_t)D * 2};
        const cuuint32_t box[2] = {64, (cuuint32_t)p.G};
        if (!encode(&maps.q, p.q, 2, dims, strides, box)) return cudaErrorInvalidValue;
    }
    {
        const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)p.Hkv, (cuuint64_t)p.B * p.S_max};
        const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)p.Hkv * D * 2};
        const cuuint32_t box[3] = {64, 1, (cuuint32_t)TcShape<D, F32>::T};
        if (!encode(&maps.k, p.k, 3, dims, strides, box)) return cudaErrorInvalidValue;
        if (!encode(&maps.v, p.v, 3, dims, strides, box)) return cudaErrorInvalidValue;
        const cuuint32_t pf_box[3] = {(cuuint32_t)D, 1, (cuuint32_t)TcShape<D, F32>::T};
        if (!encode(&maps.k_pf, p.k, 3, dims, strides, pf_box, false)) return cudaErrorInvalidValue;
        if (!encode(&maps.v_pf, p.v, 3, dims, strides, pf_box, false)) return cudaErrorInvalidValue;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.n_split, 1, 1);
    cfg.blockDim = dim3((unsigned)k.threads, 1, 1);
    cfg.dynamicSmemBytes = (size_t)k.smem_bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, split_kv_chunk_tc_kernel<D, F32>, p, maps);
}

template <int D, bool F32>
static ChunkKernel make_tc(int index) {
    using Sh = TcShape<D, F32>;
    ChunkKernel k;
    k.fn = reinterpret_cast<const void*>(split_kv_chunk_tc_kernel<D, F32>);
    k.launch = launch_tc_chunk<D, F32>;
    k.head_dim = D;
    k.threads = Sh::THREADS;
    k.smem_bytes = Sh::SMEM_BYTES;
    k.tile_tokens = Sh::T;
    k.ctas_per_sm = 1;
    k.f32_out = F32;
    k.tensor_core = true;
    k.index = index;
    return k;
}

const ChunkKernel* tc_chunk_kernel(int head_dim, bool f32_out) {
    static const ChunkKernel table[3][2] = {
        {make_tc<64, false>(6), make_tc<64, true>(7)},
        {make_tc<128, false>(8), make_tc<128, true>(9)},
        {make_tc<256, false>(10), make_tc<256, true>(11)},
    };
    const int d = head_dim == 64 ? 0 : (head_dim == 128 ? 1 : (head_dim == 256 ? 2 : -1));
    return d < 0 ? nullptr : &table[d][f32_out ? 1 : 0];
}

}  // namespace kvd
