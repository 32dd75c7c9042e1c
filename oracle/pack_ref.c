/*
 * Sequential C restatement of the packing rules, for timing the oracle on host
 * cores. TEST INFRASTRUCTURE ONLY. It shares nothing with the CUDA library; the
 * tests pin it against the literal Python oracle (oracle/pack.py) and against
 * the worked examples of the InternEvo page "Data loading and flow".
 *
 * Rules (InternEvo page "Data loading and flow", section "Dataloader loading
 * data"; fields from section "Fetching data from the Dataloader"):
 *   packed  (use_packed_dataset = 1): documents end to end, cut every
 *           plen = micro_bsz * seq_len tokens, the last row padded with 0;
 *           each document's labels are its tokens from the second on, then
 *           -100, taken before the cut.
 *   unpacked (use_packed_dataset = 0): micro_bsz documents per row, each cut
 *           to seq_len (excess dropped), labels from the cut document, the
 *           row padded with 0 / -100.
 *   segments of a row: maximal runs of one document's tokens, then the
 *           padding tail as one more segment; indexes count 0, 1, ... inside
 *           each segment; max_seqlen is the longest segment of the row.
 * Output layout is the flat one: rows concatenated; cu_seqlens global
 * (row r's boundaries + r * plen, shared row ends once); row_seg_ptr [rows+1].
 */
#include <stdint.h>
#include <stdlib.h>

/* Number of rows and an upper bound on the number of segments. */
int spd_oracle_pack_rows(int64_t num_docs, int64_t num_tokens, const int32_t *doc_lens,
                         int micro_bsz, int seq_len, int packed, int64_t *rows,
                         int64_t *max_segs)
{
    if (micro_bsz <= 0 || seq_len <= 0 || num_docs < 0) return -1;
    int64_t plen = (int64_t)micro_bsz * seq_len;
    int64_t r;
    if (packed) r = (num_tokens + plen - 1) / plen;
    else r = (num_docs + micro_bsz - 1) / micro_bsz;
    (void)doc_lens;
    *rows = r;
    *max_segs = num_docs + 2 * r;
    return 0;
}

int spd_oracle_pack(const int32_t *tokens, const int32_t *doc_lens, int64_t num_docs,
                    int64_t num_tokens, int micro_bsz, int seq_len, int packed,
                    int32_t *ids, int32_t *labels, int32_t *indexes, int32_t *cu,
                    int32_t *row_seg_ptr, int32_t *max_seqlen, int32_t *num_segs)
{
    int64_t rows, max_segs, plen = (int64_t)micro_bsz * seq_len;
    if (spd_oracle_pack_rows(num_docs, num_tokens, doc_lens, micro_bsz, seq_len, packed,
                             &rows, &max_segs))
        return -1;
    int64_t total = rows * plen, sum = 0;
    for (int64_t d = 0; d < num_docs; ++d) {
        if (doc_lens[d] <= 0) return -1;
        sum += doc_lens[d];
    }
    if (sum != num_tokens) return -1;
    int64_t *owner = (int64_t *)malloc(sizeof(int64_t) * (size_t)(total > 0 ? total : 1));
    if (!owner) return -1;
    for (int64_t p = 0; p < total; ++p) { ids[p] = 0; labels[p] = -100; owner[p] = -1; }

    if (packed) {
        int64_t p = 0, in = 0;
        for (int64_t d = 0; d < num_docs; ++d)
            for (int32_t t = 0; t < doc_lens[d]; ++t, ++p, ++in) {
                ids[p] = tokens[in];
                labels[p] = (t + 1 < doc_lens[d]) ? tokens[in + 1] : -100;
                owner[p] = d;
            }
    } else {
        int64_t in = 0, p = 0;
        for (int64_t d = 0; d < num_docs; ++d) {
            if (d % micro_bsz == 0) p = (d / micro_bsz) * plen; /* a new row starts */
            int32_t keep = doc_lens[d] < seq_len ? doc_lens[d] : seq_len;
            for (int32_t t = 0; t < keep; ++t, ++p) {
                ids[p] = tokens[in + t];
                labels[p] = (t + 1 < keep) ? tokens[in + t + 1] : -100;
                owner[p] = d;
            }
            in += doc_lens[d];
        }
    }

    int64_t ns = 0;
    cu[0] = 0;
    row_seg_ptr[0] = 0;
    for (int64_t r = 0; r < rows; ++r) {
        int64_t a = r * plen, start = a;
        int32_t mx = 0;
        for (int64_t p = a; p < a + plen; ++p) {
            int last = (p + 1 == a + plen) || owner[p + 1] != owner[p];
            indexes[p] = (int32_t)(p - start);
            if (last) {
                int32_t len = (int32_t)(p + 1 - start);
                if (len > mx) mx = len;
                cu[++ns] = (int32_t)(p + 1);
                start = p + 1;
            }
        }
        max_seqlen[r] = mx;
        row_seg_ptr[r + 1] = (int32_t)ns;
    }
    *num_segs = (int32_t)ns;
    free(owner);
    return 0;
}
