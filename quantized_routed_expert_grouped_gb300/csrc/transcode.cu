// transcode.cu - load-time transcoding of CB2/CB3 weight blobs into the slot layouts CB3X / CB2X.
//
// The idea is that of #3455 "GP100 (sm_60): 4-bit slots for resident IQ2_S / IQ3_XXS / IQ3_S
// gate/up experts", "Problem and result" / "Approach": once the weights are resident, re-encode
// the codebook formats into a layout the decode kernels read without lookups, holding the same
// values so every dot product is unchanged. Here each weight's signed odd value v = +-grid is
// stored as u = (v - 1)/2 + bias (4 bits, bias 8, for CB3X; 2 bits, bias 2, for CB2X), and the
// super-block scale D and the sub-scale nibbles are copied into an 8-byte record per 256 weights.
// A value that does not fit sets MOE_ERR_CODEBOOK; a source blob that is not 2-byte aligned or a
// destination blob that is not 8-byte aligned sets MOE_ERR_ALIGN and that blob is left unwritten.
#include "common.cuh"
#include "internal.h"

namespace moe {

// One CTA per run of R whole rows of one blob (R = 256 / chunks per row): the rows' source bytes
// are staged in shared memory with coalesced 2-byte loads, one thread per (row, 256-weight chunk)
// transcodes its chunk from there into the destination rows' image in shared memory, and the image
// goes out with coalesced 8-byte stores (a destination row is chunks x (codes + 8) bytes, a multiple
// of 8, and the rows of a run are contiguous).
__global__ void __launch_bounds__(256) transcode_kernel(int src_type, const int8_t* __restrict__ cb, int dst_type,
                                                        int K, int rows, int R, const void* const* src_blobs,
                                                        void* const* dst_blobs, int32_t* err) {
    extern __shared__ __align__(16) uint8_t tsm[];
    const int nch = K / 256;
    const bool cb3 = src_type == MOE_CB3;
    const int src_chunk = cb3 ? 102 : 70;
    const int code_bytes = dst_type == MOE_CB3X ? 128 : 64;
    const int src_rb = nch * src_chunk, dst_rb = nch * (code_bytes + 8);
    const int b = blockIdx.y, r0 = blockIdx.x * R;
    const int nr = rows - r0 < R ? rows - r0 : R;
    if (nr <= 0) return;
    // the staging loads are 2 bytes wide and the stores 8: a blob off those boundaries is skipped
    if ((reinterpret_cast<uintptr_t>(src_blobs[b]) & 1) || (reinterpret_cast<uintptr_t>(dst_blobs[b]) & 7)) {
        if (threadIdx.x == 0) set_err(err, MOE_ERR_ALIGN);  // the blob is skipped
        return;
    }
    uint8_t* ssrc = tsm;                                   // [R][src_rb]
    uint8_t* sdst = tsm + ((R * src_rb + 15) & ~15);      // [R][dst_rb]
    const uint8_t* gsrc = static_cast<const uint8_t*>(src_blobs[b]) + static_cast<size_t>(r0) * src_rb;
    uint8_t* gdst = static_cast<uint8_t*>(dst_blobs[b]) + static_cast<size_t>(r0) * dst_rb;
    // the run's source bytes (src_rb is even: 2-byte loads are aligned)
    {
        const uint16_t* g2 = reinterpret_cast<const uint16_t*>(gsrc);
        uint16_t* s2 = reinterpret_cast<uint16_t*>(ssrc);
        for (int i = threadIdx.x; i < nr * src_rb / 2; i += blockDim.x) s2[i] = __ldg(g2 + i);
    }
    __syncthreads();
    const int ri = threadIdx.x / nch, c = threadIdx.x - ri * nch;
    if (ri < nr) {
        const int bias = dst_type == MOE_CB3X ? 8 : 2, umax = dst_type == MOE_CB3X ? 15 : 3;
        const uint8_t* sb = ssrc + ri * src_rb + c * src_chunk;
        uint8_t* drow = sdst + ri * dst_rb;
        uint32_t words[32];  // the chunk's codes (128 or 64 bytes)
        for (int k = 0; k < 32; ++k) words[k] = 0;
        bool bad = false;
        for (int n = 0; n < 256; ++n) {
            int v;
            if (cb3) {
                v = cb[sb[2 + n / 4] * 4 + (n % 4)];
                if ((sb[66 + n / 8] >> (n % 8)) & 1) v = -v;
            } else {
                v = cb[sb[2 + n / 8] * 8 + (n % 8)];
                if ((sb[34 + n / 8] >> (n % 8)) & 1) v = -v;
            }
            int u = ((v - 1) >> 1) + bias;  // v odd: (v - 1) is even, the shift is exact
            if ((v & 1) == 0 || u < 0 || u > umax) {
                bad = true;
                u = 0;
            }
            const int j = n / 32, w = n % 32;
            int byte, shift;
            if (dst_type == MOE_CB3X) {  // sub-block j: byte w (low nibble) or w-16 (high nibble)
                byte = j * 16 + (w & 15);
                shift = w < 16 ? 0 : 4;
            } else {  // sub-block j: byte w%8, bits 2*(w/8)
                byte = j * 8 + (w & 7);
                shift = 2 * (w >> 3);
            }
            words[byte >> 2] |= static_cast<uint32_t>(u) << (8 * (byte & 3) + shift);
        }
        uint32_t* dc = reinterpret_cast<uint32_t*>(drow + c * code_bytes);
        for (int k = 0; k < code_bytes / 4; ++k) dc[k] = words[k];
        uint8_t* rec = drow + nch * code_bytes + c * 8;
        const uint8_t* sub = sb + (cb3 ? 98 : 66);
        rec[0] = sb[0];
        rec[1] = sb[1];
        rec[2] = 0;
        rec[3] = 0;
        for (int k = 0; k < 4; ++k) rec[4 + k] = sub[k];
        if (bad) set_err(err, MOE_ERR_CODEBOOK);
    }
    __syncthreads();
    // the run's destination image, 8 bytes at a time
    {
        const uint2* s8 = reinterpret_cast<const uint2*>(sdst);
        uint2* g8 = reinterpret_cast<uint2*>(gdst);
        for (int i = threadIdx.x; i < nr * dst_rb / 8; i += blockDim.x) g8[i] = s8[i];
    }
}

cudaError_t launch_transcode_cb(int src_type, const int8_t* codebook, int dst_type, int K, int rows, int n_blobs,
                                const void* const* src_blobs, void* const* dst_blobs, int32_t* err, cudaStream_t s) {
    const int nch = K / 256;
    if (nch <= 0 || nch > 256 || n_blobs > 65535) return cudaErrorInvalidValue;
    const int R = 256 / nch > 0 ? 256 / nch : 1;  // whole rows per CTA
    const int src_rb = nch * (src_type == MOE_CB3 ? 102 : 70);
    const int dst_rb = nch * ((dst_type == MOE_CB3X ? 128 : 64) + 8);
    const int smem = ((R * src_rb + 15) & ~15) + R * dst_rb;
    cudaError_t e = cudaFuncSetAttribute(transcode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const dim3 grid(static_cast<unsigned>((rows + R - 1) / R), static_cast<unsigned>(n_blobs));
    return launch_kernel(transcode_kernel, grid, dim3(static_cast<unsigned>(R * nch)), static_cast<size_t>(smem), s,
                         false, src_type, codebook, dst_type, K, rows, R, src_blobs, dst_blobs, err);
}

}  // namespace moe
