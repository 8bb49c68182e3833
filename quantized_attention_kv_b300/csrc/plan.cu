// plan.cu -- record layout of one (head, tensor) and the decoder's read plan.
//
// The pages fix only that every token takes the same number of bits ("Spend
// Bits Where Queries Look", Abstract: fixed per-token bit count).  The layout
// used here: each code is stored whole, least significant bit first, in
// consecutive record bits; the channels with b_j > 0 follow one another in
// the order given by this rule --
//     p2 = p1 = 8;  repeat: need = 7 - p2 - p1;  take the narrowest remaining
//     channel of width >= need (lowest index on ties), or the widest remaining
//     one if none is that wide (lowest index on ties);  p2 = p1, p1 = width.
// The rule mixes wide and narrow codes so that a byte rarely holds parts of
// more than four codes, which the fast decoder needs.
//
// The read plan cuts every byte into its pieces (the parts of the codes lying
// in it, in increasing bit position) and turns them into AND masks: see
// HeadPlan in internal.h.
#include <string.h>

#include <vector>

#include "internal.h"

namespace {

constexpr int D = AATC_D;

struct Piece {
    int ch;    // channel
    int o;     // first code bit held by the piece
    int n;     // width
    int p;     // bit position inside its byte
};

int record_order(const int32_t *bits, int *order)
{
    bool used[D] = {};
    int total = 0, n = 0, p2 = 8, p1 = 8;
    for (int j = 0; j < D; ++j) total += bits[j] > 0;
    while (n < total) {
        const int need = 7 - p2 - p1;
        int pick = -1, widest = -1;
        for (int j = 0; j < D; ++j) {
            if (used[j] || bits[j] <= 0) continue;
            if (bits[j] >= need && (pick < 0 || bits[j] < bits[pick])) pick = j;
            if (widest < 0 || bits[j] > bits[widest]) widest = j;
        }
        if (pick < 0) pick = widest;
        used[pick] = true;
        order[n++] = pick;
        p2 = p1;
        p1 = bits[pick];
    }
    return n;
}

}  // namespace

// kp: pieces per byte the read plan provides (4 or 8); no masks when a byte
// holds more
void plan_one(const int32_t *bits, int W, int kp, HeadPlan *out)
{
    memset(out, 0, sizeof(*out));
    for (int j = 0; j < D; ++j) out->off[j] = -1;
    for (int s = 0; s < AATC_PLAN_SLOTS; ++s)
        for (int k = 0; k < 16; ++k) out->ch[s][k][0] = out->ch[s][k][1] = -1;

    int order[D];
    const int n = record_order(bits, order);
    out->n_coded = n;
    for (int a = 0; a < D; ++a) out->order[a] = (int16_t)(a < n ? order[a] : -1);
    const int nbytes = 4 * W;
    std::vector<std::vector<Piece>> by(nbytes);
    int pos = 0;
    for (int a = 0; a < n; ++a) {
        const int j = order[a];
        out->off[j] = (int16_t)pos;
        int o = 0, w = bits[j];
        while (w > 0) {
            const int byte = pos / 8, p = pos % 8;
            const int take = w < 8 - p ? w : 8 - p;
            if (byte < nbytes) by[byte].push_back(Piece{j, o, take, p});
            pos += take;
            o += take;
            w -= take;
        }
    }
    int mp = 0;
    for (int b = 0; b < nbytes; ++b) mp = (int)by[b].size() > mp ? (int)by[b].size() : mp;
    out->max_pieces = mp;
    if (mp > kp) return;   // no read plan at kp pieces per byte

    auto piece = [&](int byte, int k) -> const Piece * {
        return (byte < nbytes && k < (int)by[byte].size()) ? &by[byte][k] : nullptr;
    };
    auto fmask = [](const Piece *pc) -> uint32_t {
        return pc ? (((1u << pc->n) - 1u) << pc->p) : 0u;
    };
    // keys: record word w, slot k < 2 kp; low half from byte 4w (+1 for
    // slots k >= kp), high half from byte 4w+2 (+1)
    for (int w = 0; w < W && w < AATC_PLAN_SLOTS; ++w)
        for (int k = 0; k < 2 * kp; ++k) {
            const int sb = k < kp ? 0 : 1, pk = k % kp;
            const Piece *lo = piece(4 * w + sb, pk), *hi = piece(4 * w + 2 + sb, pk);
            out->mask[w][k] = fmask(lo) | (fmask(hi) << 16);
            if (lo) { out->ch[w][k][0] = (int8_t)lo->ch; out->ex[w][k][0] = (int8_t)(lo->o - lo->p); }
            if (hi) { out->ch[w][k][1] = (int8_t)hi->ch; out->ex[w][k][1] = (int8_t)(hi->o - hi->p); }
        }
}

aatc_status plan_build(aatc_calib *h, const int32_t *bits_k, const int32_t *bits_v)
{
    std::vector<HeadPlan> plans((size_t)h->Hkv * 2);
    bool fast = true;
    // keys: 4 pieces per byte, or 8 for every head when a key byte of some head holds more than 4
    int kp = AATC_PIECES;
    for (int hh = 0; hh < h->Hkv; ++hh) {
        plan_one(bits_k + (size_t)hh * D, h->Wk, AATC_PIECES, &plans[hh * 2 + 0]);
        if (plans[hh * 2].max_pieces > AATC_PIECES) kp = AATC_KEY_PIECES;
    }
    h->kpieces = kp;
    for (int hh = 0; hh < h->Hkv; ++hh) {
        if (kp != AATC_PIECES) plan_one(bits_k + (size_t)hh * D, h->Wk, kp, &plans[hh * 2 + 0]);
        // values: the same cut into pieces, read per half-word (slot = half-word e,
        // mask in both halves: the pair word holds half-word e of two tokens)
        HeadPlan key_view;
        plan_one(bits_v + (size_t)hh * D, h->Wv, AATC_PIECES, &key_view);
        fast = fast && plans[hh * 2].max_pieces <= kp && key_view.max_pieces <= AATC_PIECES;
        HeadPlan &pv = plans[hh * 2 + 1];
        memcpy(&pv, &key_view, sizeof(HeadPlan));
        for (int s = 0; s < AATC_PLAN_SLOTS; ++s)
            for (int k = 0; k < 16; ++k) {
                pv.mask[s][k] = 0;
                pv.ch[s][k][0] = pv.ch[s][k][1] = -1;
                pv.ex[s][k][0] = pv.ex[s][k][1] = 0;
            }
        if (key_view.max_pieces <= AATC_PIECES) {
            // half-word e = bytes 2e (S = 0) and 2e+1 (S = 1); record word e/2 holds
            // them at bytes 2(e%2) and 2(e%2)+1, i.e. in key_view's slot of word e/2:
            // low half (e even) or high half (e odd)
            for (int e = 0; e < 2 * h->Wv && e < AATC_PLAN_SLOTS; ++e)
                for (int k = 0; k < 8; ++k) {
                    const int w = e / 2, half = e % 2;
                    const uint32_t m = (key_view.mask[w][k] >> (16 * half)) & 0xFFFFu;
                    pv.mask[e][k] = m | (m << 16);
                    pv.ch[e][k][0] = key_view.ch[w][k][half];
                    pv.ex[e][k][0] = key_view.ex[w][k][half];
                }
        }
    }
    h->fast_layout = fast;
    AATC_CUDA(cudaMemcpy(h->plan, plans.data(), sizeof(HeadPlan) * plans.size(), cudaMemcpyHostToDevice));
    aatc_status st = enc_build(h, 0);
    if (st == AATC_OK) st = dec_build(h, 0);
    if (st == AATC_OK) AATC_CUDA(cudaDeviceSynchronize());
    return st;
}
