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

template <int D, bool F32, int QR>
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
        const cuuint32_t box[3] = {64, 1, (cuuint32_t)TcShape<D, F32, QR>::T};
        if (!encode(&maps.k, p.k, 3, dims, strides, box)) return cudaErrorInvalidValue;
        if (!encode(&maps.v, p.v, 3, dims, strides, box)) return cudaErrorInvalidValue;
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
    return cudaLaunchKernelEx(&cfg, split_kv_chunk_tc_kernel<D, F32, QR>, p, maps);
}

template <int D, bool F32, int QR>
static ChunkKernel make_tc(int index) {
    using Sh = TcShape<D, F32, QR>;
    ChunkKernel k;
    k.fn = reinterpret_cast<const void*>(split_kv_chunk_tc_kernel<D, F32, QR>);
    k.launch = launch_tc_chunk<D, F32, QR>;
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

// Groups of up to 48 query heads store Q in 48-row blocks (saving shared
// memory for a third K stage); wider groups in 64-row blocks.
const ChunkKernel* tc_chunk_kernel(int head_dim, bool f32_out, int group) {
    static const ChunkKernel table[3][2][2] = {
        {{make_tc<64, false, 48>(6), make_tc<64, true, 48>(7)}, {make_tc<64, false, 64>(8), make_tc<64, true, 64>(9)}},
        {{make_tc<128, false, 48>(10), make_tc<128, true, 48>(11)},
         {make_tc<128, false, 64>(12), make_tc<128, true, 64>(13)}},
        {{make_tc<256, false, 48>(14), make_tc<256, true, 48>(15)},
         {make_tc<256, false, 64>(16), make_tc<256, true, 64>(17)}},
    };
    const int d = head_dim == 64 ? 0 : (head_dim == 128 ? 1 : (head_dim == 256 ? 2 : -1));
    if (d < 0 || group < 1 || group > 64) return nullptr;
    return &table[d][group <= 48 ? 0 : 1][f32_out ? 1 : 0];
}

}  // namespace kvd
