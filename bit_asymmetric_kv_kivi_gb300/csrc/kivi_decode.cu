// Decode attention: the split policy and workspace plan, and the dispatch over the key
// and value code widths to the kernels of kivi_decode_impl.cuh (one translation unit
// per pair of widths).
#include "kivi_internal.cuh"

namespace kivi {

// Tickets at the start of every workspace: one int32 per stream, with room for two streams
// per kv head in every plan. Decode and multi-query calls may then share one workspace:
// every plan's records start past the tickets of any plan, and every kernel leaves its
// tickets at zero (the last CTA of a stream resets its ticket).
static size_t ticket_bytes(int nseq, int H) {
    return ((2 * static_cast<size_t>(nseq) * H * sizeof(int32_t) + 255) / 256) * 256;
}

void mma_plan(int nseq, int H, int D, int per, int streams_per_kv_head, size_t* counter_bytes, size_t* partial_bytes) {
    // decode_mma_kernel over streams of `per` query heads, streams_per_kv_head per (sequence,
    // kv head): one record of `per` heads per segment, fewer than 2 S + kDecodeMaxCtas of them.
    // The tickets in front are the multi-query kernel's; this kernel takes none.
    const size_t S = static_cast<size_t>(nseq) * H * streams_per_kv_head;
    *counter_bytes = ticket_bytes(nseq, H);
    *partial_bytes = (2 * S + kDecodeMaxCtas) * per * (D + 4) * sizeof(float);
}

void decode_plan(int nseq, int H, int Hq, int D, int max_kv_len, int* chunk, int* max_splits,
                 size_t* counter_bytes, size_t* partial_bytes) {
    const int gq = H > 0 ? Hq / H : 0;
    if (gq == 1 || gq == 2 || gq == 4 || gq == 8) {
        // the persistent kernel, one stream of gq heads per kv head
        *chunk = 0;
        *max_splits = 0;
        mma_plan(nseq, H, D, gq, 1, counter_bytes, partial_bytes);
        return;
    }
    // other query groups (up to 32): decode_multi_kernel with one query per sequence
    multi_plan(nseq, H, Hq, D, 1, max_kv_len, chunk, max_splits, counter_bytes, partial_bytes);
}

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream) {
    if (a.nseq == 0) return cudaSuccess;
    const int gq = a.Hq / a.H;
    // multi-query calls reach here only with one query, with up to 32 / gq queries at a query
    // group of 4 or 8, or with two queries at a group of 1 or 2 (one stream of gq heads per
    // query and kv head)
    if (a.n_query > 1 && !(((gq == 4 || gq == 8) && a.n_query * gq <= 32) || ((gq == 1 || gq == 2) && a.n_query == 2)))
        return cudaErrorInvalidValue;
    if (gq != 1 && gq != 2 && gq != 4 && gq != 8) {
        DecodeArgs m = a;
        m.n_query = 0;     // decode: one query per sequence, empty sequences give zeros
        return launch_multi(m, stream);
    }
    if (a.kb == 2) return a.vb == 2 ? launch_decode_k2v2(a, stream) : launch_decode_k2v4(a, stream);
    return a.vb == 2 ? launch_decode_k4v2(a, stream) : launch_decode_k4v4(a, stream);
}

// Multi-query attention: packed splits of a whole number of 32-token tiles, about an eighth
// of the longest sequence in 256-token steps between 1024 and 4096 tokens, plus one split
// for the residual window; one record of kD + 4 floats per (split, virtual head), the
// virtual heads padded to whole warps of four.
void multi_plan(int nseq, int H, int Hq, int D, int n_query, int max_kv_len, int* chunk, int* max_splits,
                size_t* counter_bytes, size_t* partial_bytes) {
    *counter_bytes = ticket_bytes(nseq, H);
    const int V = H > 0 ? n_query * (Hq / H) : 0;
    const int w = V <= 4 ? 1 : V <= 8 ? 2 : V <= 16 ? 4 : 8;
    const int64_t eighth = (static_cast<int64_t>(max_kv_len) + 7) / 8;
    int64_t c = ((eighth + 255) / 256) * 256;
    c = c < 1024 ? 1024 : (c > 4096 ? 4096 : c);
    const int64_t ms = (max_kv_len <= 0 ? 0 : (max_kv_len + c - 1) / c) + 1;
    *chunk = static_cast<int>(c);
    *max_splits = static_cast<int>(ms);
    *partial_bytes = static_cast<size_t>(nseq) * H * ms * (4 * w) * (D + 4) * sizeof(float);
}

cudaError_t launch_multi(const DecodeArgs& a, cudaStream_t stream) {
    if (a.nseq == 0) return cudaSuccess;
    if (a.kb == 2) return a.vb == 2 ? launch_multi_k2v2(a, stream) : launch_multi_k2v4(a, stream);
    return a.vb == 2 ? launch_multi_k4v2(a, stream) : launch_multi_k4v4(a, stream);
}

}  // namespace kivi
