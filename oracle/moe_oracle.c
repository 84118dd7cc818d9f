/*
 * CPU oracle for the routing metadata of the MoE expert-parallel layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or calls this
 * file; only the tests, the package smoke check and the benchmark's CPU-baseline leg do.
 * It shares no code, header or table with the CUDA path.
 *
 * It is the plain definition written out as literal loops over the picks (t, j) in
 * lexicographic order, following:
 *   - Mooncake EP guide, "Buffer.dispatch(...)": topk_idx [num_tokens, top_k], -1 marks a
 *     masked pick; num_experts must divide by the number of ranks; the dispatch output
 *     is the local-expert-major packed layout [num_local_experts, num_ranks*max_tok,
 *     hidden] with packed_recv_count, packed_recv_src_info, packed_recv_layout_range.
 *   - FlashInfer MoE-EP page, section 3 "Algorithm / layout contracts": EXPERT_MAJOR rows
 *     are pre-assigned to experts; RANK_MAJOR receives [world, max_tok, hidden] grouped by
 *     source rank; HT FLAT receives [num_recv, hidden] token-major; received topk_idx are
 *     LOCAL expert indices with -1 for non-local picks.
 * Readings where the pages are silent (stated once, used throughout):
 *   - order inside an expert region / a receive region is ascending (token, pick);
 *   - a token is received by destination rank d once if any of its valid picks lives on d;
 *   - an id outside [-1, E) is an error: it is counted and the pick is dropped;
 *   - EP rank-health mask (Mooncake EP guide, Buffer.dispatch `active_ranks`, int32
 *     [num_ranks], 0 = failed rank; "Active-rank tensors: PG vs EP"): a pick is dropped
 *     when its expert lives on an inactive rank or its token belongs to an inactive source
 *     rank (`active` NULL = all ranks active).
 */

#include <stdint.h>

/* 1 iff pick (t, e) survives the rank-health mask. */
static int rank_ok(const int32_t *active, int Le, int Tr, int t, int64_t e)
{
    if (!active) return 1;
    return active[e / Le] != 0 && active[t / Tr] != 0;
}

/* Expert-grouped pick list (shared by all three layouts).
 *   cap          capacity of one expert's region in rows, or -1 for no limit.  The
 *                EXPERT_MAJOR region of an expert holds num_ranks * max_tok rows, which
 *                every token can fill at most once per distinct expert; a token naming
 *                the same expert twice could overflow it.  A pick whose rank inside its
 *                expert reaches cap is dropped (not dispatched, computed or combined)
 *                and counted in *n_over.
 *   counts[e]    number of kept picks of expert e
 *   offsets[e]   sum of counts[e'] for e' < e (offsets[E] = R, the number of kept picks)
 *   pick_pos[i]  for pick i = t*k + j: offsets[e] + #{earlier kept picks of e}, or -1
 *   pick_src[p]  inverse of pick_pos on kept picks
 *   layout_range[(e*W + r)*2 + {0,1}]  (begin inside expert e's region, count) of the
 *                kept picks whose token belongs to source rank r = t / Tr
 * Returns the number of ids outside [-1, E).
 */
int oracle_route_experts(int T, int k, int E, int W, int Tr, int64_t cap, const int64_t *ids,
                         const int32_t *active, int32_t *counts, int32_t *offsets,
                         int32_t *pick_pos, int32_t *pick_src, int32_t *layout_range,
                         int32_t *n_over, int32_t *n_inactive)
{
    int bad = 0;
    int Le = E / W;
    *n_over = 0;
    *n_inactive = 0;
    for (int e = 0; e < E; ++e) counts[e] = 0;
    for (int i = 0; i < E * W * 2; ++i) layout_range[i] = 0;
    for (int t = 0; t < T; ++t)
        for (int j = 0; j < k; ++j) {
            int64_t e = ids[(int64_t)t * k + j];
            if (e == -1) continue;
            if (e < -1 || e >= E) { ++bad; continue; }
            if (!rank_ok(active, Le, Tr, t, e)) { *n_inactive += 1; continue; }
            if (cap >= 0 && counts[e] >= cap) { *n_over += 1; continue; }
            counts[e] += 1;
            layout_range[(e * W + t / Tr) * 2 + 1] += 1;
        }
    offsets[0] = 0;
    for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
    for (int e = 0; e < E; ++e) {
        int begin = 0;
        for (int r = 0; r < W; ++r) {
            layout_range[(e * W + r) * 2 + 0] = begin;
            begin += layout_range[(e * W + r) * 2 + 1];
        }
    }
    /* next free position of every expert, walked in (t, j) order */
    int32_t next[E > 0 ? E : 1];
    for (int e = 0; e < E; ++e) next[e] = offsets[e];
    for (int t = 0; t < T; ++t)
        for (int j = 0; j < k; ++j) {
            int64_t i = (int64_t)t * k + j;
            int64_t e = ids[i];
            if (e < 0 || e >= E || !rank_ok(active, Le, Tr, t, e) || next[e] == offsets[e + 1]) {
                pick_pos[i] = -1;
                continue;
            }
            int p = next[e]++;
            pick_pos[i] = p;
            pick_src[p] = (int32_t)i;
        }
    return bad;
}

/* Destination-rank receive metadata for RANK_MAJOR (layout 1) and FLAT (layout 2).
 * Each destination d owns a region of cap = W*Tr rows.
 *   recv_row[t*W + d]   row of token t inside d's region, or -1 if t has no pick on d
 *                       RANK_MAJOR: s*Tr + #{earlier tokens of source rank s received by d}
 *                       FLAT:       #{earlier tokens received by d}
 *   recv_count[d*W + s] tokens of source rank s received by d
 *   num_recv[d]         tokens received by d
 *   recv_src[d*cap + row]            token index of that row (rows that hold a token)
 *   recv_topk_idx[(d*cap+row)*k + j] local expert id e - d*Le if pick j lives on d, else -1
 *   recv_topk_w[(d*cap+row)*k + j]   topk_weights[t, j] if pick j lives on d, else 0
 */
void oracle_route_ranks(int T, int k, int E, int W, int Tr, int layout,
                        const int64_t *ids, const int32_t *active, const float *topk_w,
                        int32_t *recv_row, int32_t *recv_count, int32_t *num_recv,
                        int32_t *recv_src, int32_t *recv_topk_idx, float *recv_topk_w)
{
    int Le = E / W;
    int64_t cap = (int64_t)W * Tr;
    for (int i = 0; i < W * W; ++i) recv_count[i] = 0;
    for (int d = 0; d < W; ++d) num_recv[d] = 0;
    for (int t = 0; t < T; ++t) {
        int s = t / Tr;
        for (int d = 0; d < W; ++d) {
            int on_d = 0;
            for (int j = 0; j < k; ++j) {
                int64_t e = ids[(int64_t)t * k + j];
                if (e >= 0 && e < E && e / Le == d && rank_ok(active, Le, Tr, t, e)) on_d = 1;
            }
            if (!on_d) { recv_row[(int64_t)t * W + d] = -1; continue; }
            int row = (layout == 1) ? s * Tr + recv_count[d * W + s] : num_recv[d];
            recv_count[d * W + s] += 1;
            num_recv[d] += 1;
            recv_row[(int64_t)t * W + d] = row;
            recv_src[d * cap + row] = t;
            for (int j = 0; j < k; ++j) {
                int64_t e = ids[(int64_t)t * k + j];
                int64_t o = (d * cap + row) * k + j;
                if (e >= 0 && e < E && e / Le == d && rank_ok(active, Le, Tr, t, e)) {
                    recv_topk_idx[o] = (int32_t)(e - (int64_t)d * Le);
                    recv_topk_w[o] = topk_w[(int64_t)t * k + j];
                } else {
                    recv_topk_idx[o] = -1;
                    recv_topk_w[o] = 0.0f;
                }
            }
        }
    }
}
