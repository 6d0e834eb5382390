// The pair list of one rank in a ring of ranks (host only).
//
// Page: "Sequence parallelism -- splitting the token dimension across GPUs"
// (llmdaily, day 58).  "A better mental model: move blocks past the queries":
// each GPU keeps its queries; in round r+1 GPU i holds the K/V block that
// started on GPU (i - r) mod N, then passes it on.  "Causal attention gives us
// another optimization": a query block never needs keys that all come after
// it, so such pairs are skipped -- which, with contiguous chunks, leaves the
// last rank with N blocks of work and the first with one.
//
// The zigzag layout evens that out: with S = T/(2N), rank i owns pieces i and
// 2N-1-i.  In round 0 a rank attends its own two pieces (two diagonal
// blocks and one full block); in every later round exactly two full S x S
// blocks are needed -- both of its pieces against the lower piece of the
// source rank when the source is an earlier rank, or its upper piece against
// both of the source's pieces when the source is a later rank.
//
// Each query piece's pairs are numbered in execution order: the first one
// writes the accumulator, the middle ones merge into it, the last one merges
// and writes the output; a piece with a single pair writes the output
// directly.
#include <vector>

#include "rsa_internal.h"

using rsa::fail;

namespace {

struct Piece {
    int64_t row0, pos, len;
};

// The pieces rank r owns, in buffer order.
std::vector<Piece> pieces(int N, int r, int64_t T, int layout)
{
    std::vector<Piece> out;
    if (layout == RSA_LAYOUT_CONTIGUOUS) {
        const int64_t Tc = T / N;
        out.push_back(Piece{0, r * Tc, Tc});
    } else {
        const int64_t S = T / (2 * N);
        out.push_back(Piece{0, r * S, S});
        out.push_back(Piece{S, (int64_t)(2 * N - 1 - r) * S, S});
    }
    return out;
}

}  // namespace

extern "C" rsa_status rsa_rank_ring_plan(int N, int rank, int64_t T, int causal, int layout, int64_t *steps,
                                         int cap, int *n_steps)
{
    if (!n_steps)
        return fail(RSA_ERR_INVALID_ARG, "n_steps is NULL");
    *n_steps = 0;
    if (N < 1 || N > 4096 || rank < 0 || rank >= N || T < 1)
        return fail(RSA_ERR_INVALID_ARG, "need 1 <= N <= 4096, 0 <= rank < N, T >= 1");
    if (layout != RSA_LAYOUT_CONTIGUOUS && layout != RSA_LAYOUT_ZIGZAG)
        return fail(RSA_ERR_INVALID_ARG, "layout %d is not RSA_LAYOUT_CONTIGUOUS or RSA_LAYOUT_ZIGZAG", layout);
    const int64_t parts = layout == RSA_LAYOUT_ZIGZAG ? 2 * (int64_t)N : N;
    if (T % parts != 0)
        return fail(RSA_ERR_INVALID_ARG, "T=%lld must be a multiple of %lld for this layout", (long long)T,
                    (long long)parts);
    struct Step {
        int round, src, qp;  // qp: which of this rank's pieces
        Piece q, kv;
    };
    const std::vector<Piece> mine = pieces(N, rank, T, layout);
    std::vector<Step> plan;
    for (int r = 0; r < N; ++r) {
        const int src = ((rank - r) % N + N) % N;
        const std::vector<Piece> theirs = pieces(N, src, T, layout);
        for (int a = 0; a < (int)mine.size(); ++a)
            for (const Piece &kv : theirs) {
                const Piece &q = mine[a];
                if (causal && kv.pos > q.pos + q.len - 1)
                    continue;  // every key after every query of the piece
                plan.push_back(Step{r, src, a, q, kv});
            }
    }
    *n_steps = (int)plan.size();
    if ((int)plan.size() > cap || (!plan.empty() && !steps))
        return fail(RSA_ERR_INVALID_ARG, "the plan has %zu steps; cap=%d", plan.size(), cap);
    // fold mode: position of the step among its query piece's steps
    std::vector<int> total(mine.size(), 0), seen(mine.size(), 0);
    for (const Step &s : plan)
        ++total[s.qp];
    for (size_t i = 0; i < plan.size(); ++i) {
        const Step &s = plan[i];
        const int k = seen[s.qp]++;
        const int n = total[s.qp];
        const int fold = n == 1 ? RSA_FOLD_ONLY : (k == 0 ? RSA_FOLD_FIRST : (k == n - 1 ? RSA_FOLD_LAST : RSA_FOLD_MERGE));
        int64_t *o = steps + 9 * i;
        o[0] = s.round;
        o[1] = s.src;
        o[2] = s.q.row0;
        o[3] = s.q.pos;
        o[4] = s.q.len;
        o[5] = s.kv.row0;
        o[6] = s.kv.pos;
        o[7] = s.kv.len;
        o[8] = fold;
    }
    return RSA_OK;
}
