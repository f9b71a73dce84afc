/*
 * CPU oracle for bit-exact delta-compressed refit.  TEST INFRASTRUCTURE ONLY
 * (see oracle.h): loaded by the test suite, the smoke check and the
 * benchmark's CPU-baseline leg, never by the product path.
 *
 * Plain, slow, obviously correct: canonicalisation and receiver placement by
 * explicit per-element index loops, bytewise XOR, per-element change counts,
 * a greedy LZ4 block encoder and a strict decoder written from the public LZ4
 * block format, scalar apply.  Chunks run in parallel (one pthread pool over
 * independent 64 KiB chunks); nothing else is reordered or fused.
 *
 * Sources (the four pages on NeMo-DCR and GPU weight teleportation):
 *   [P1] NeMo-DCR paper summary, "Method": change detection per owner shard,
 *        direct projection, residual conversion, hybrid encoding, recoverable
 *        in-place apply with retry and joint commit.
 *   [P2] Popular write-up, sections on canonical coordinates, shard owners
 *        (bitwise compare, +0 vs -0), XOR versus overwrite, dedup by unique
 *        IDs, in-place apply without a backup and overwrite-only retry.
 *   [P3] Paper abstract (Italian translation): XOR masks for affine changes,
 *        overwrites for the rest, retries overwrite partial writes.
 *   [P4] "GPU-accelerated weight teleportation", sections "Delta update
 *        algebra" (mask = old XOR new), "A strong baseline with the
 *        Blackwell-native DE" (LZ4 block format, CPU-prepared apply plan) and
 *        "Working with low-precision RL" (layout remap of gate/up rows paired
 *        in groups of 64).
 * Where the pages are silent this file takes the plainest reading:
 *   - chunks are 64 KiB of each canonical tensor's own row-major bytes and
 *     never straddle tensors (the last one of a tensor may be short);
 *   - a changed stored value is an element of the stored width (bf16 word,
 *     e4m3 byte, e2m1 nibble, low nibble first) whose bits differ;
 *   - the LZ4 encoder is a plain greedy one: a 2^14-slot table of the latest
 *     position per multiplicative hash of the 4-byte little-endian word,
 *     every position inserted, matches extended forward only;
 *   - windows pack whole tensors in order up to the window size, and a
 *     tensor larger than a window is cut at chunk boundaries;
 *   - the wire format (stream header, 16-byte-aligned frames with 32-byte
 *     headers in ascending chunk order, a trailing index of frame offsets)
 *     is the library's, restated here from its description.
 */
#include <pthread.h>
#include <stdatomic.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include "oracle.h"

/* ------------------------------------------------------------------------ */
/* canonical parts: one per tensor, three (q, k, v) for a fused QKV tensor   */
/* ------------------------------------------------------------------------ */
typedef struct {
    uint32_t desc, sub, residual, bits;
    uint64_t rows, cols, bytes, recv_off;
    uint64_t chunk0, nchunks;
} part_t;

typedef struct {
    part_t* parts;
    uint64_t n_parts, n_chunks, n_windows, canonical_bytes, hash;
    uint64_t* win_start;    /* n_windows + 1 chunk ids */
    uint64_t* chunk_part;   /* chunk -> part index */
} layout_t;

static void layout_free(layout_t* L)
{
    free(L->parts);
    free(L->win_start);
    free(L->chunk_part);
    memset(L, 0, sizeof(*L));
}

static int desc_ok(const orc_tensor* d)
{
    if (d->elem_bits != 4 && d->elem_bits != 8 && d->elem_bits != 16) return 0;
    if (d->tp < 1 || d->tp > ORC_MAX_TP || d->rows == 0 || d->cols == 0) return 0;
    if (d->elem_bits == 4 && d->cols % 2) return 0;
    switch (d->split) {
    case ORC_REPLICATED: break;
    case ORC_SPLIT_ROWS: if (d->rows % d->tp) return 0; break;
    case ORC_SPLIT_COLS:
        if (d->cols % d->tp) return 0;
        if (d->elem_bits == 4 && (d->cols / d->tp) % 2) return 0;
        break;
    case ORC_RESIDUAL_QKV:
        if (!d->q_heads || !d->kv_heads || !d->head_dim) return 0;
        if (d->q_heads % d->kv_heads || d->kv_heads % d->tp) return 0;
        if (d->rows != (uint64_t)(d->q_heads + 2 * d->kv_heads) * d->head_dim) return 0;
        if (d->recv_layout != ORC_RECV_CANONICAL) return 0;
        break;
    default: return 0;
    }
    if (d->recv_layout == ORC_RECV_ROWGROUP) {
        if (!d->recv_group || d->rows % d->recv_group || d->recv_slot > 1) return 0;
    } else if (d->recv_layout != ORC_RECV_CANONICAL) {
        return 0;
    }
    return 1;
}

/* FNV-1a 64 over the canonical description both ends must agree on. */
static void fnv(uint64_t* h, const void* p, size_t n)
{
    const uint8_t* b = (const uint8_t*)p;
    for (size_t i = 0; i < n; ++i) {
        *h ^= b[i];
        *h *= 0x100000001B3ULL;
    }
}
static void fnv32(uint64_t* h, uint32_t v)
{
    uint8_t b[4] = {(uint8_t)v, (uint8_t)(v >> 8), (uint8_t)(v >> 16), (uint8_t)(v >> 24)};
    fnv(h, b, 4);
}
static void fnv64(uint64_t* h, uint64_t v)
{
    fnv32(h, (uint32_t)v);
    fnv32(h, (uint32_t)(v >> 32));
}

uint64_t orc_fnv1a64(const uint8_t* p, uint64_t n)
{
    uint64_t h = 0xCBF29CE484222325ULL;
    fnv(&h, p, (size_t)n);
    return h;
}

/* Chunks: each canonical part is cut into 64 KiB pieces of its own byte
 * space (a part's last chunk may be short).  Windows: whole tensors are
 * packed in order while the window stays within window_bytes; a tensor larger
 * than a window is split at chunk boundaries. */
static int layout_build(const orc_tensor* t, uint32_t n, uint64_t window_bytes, layout_t* L)
{
    memset(L, 0, sizeof(*L));
    if (!t || n == 0 || window_bytes < ORC_CHUNK) return ORC_E_INVALID;
    uint64_t np = 0;
    for (uint32_t i = 0; i < n; ++i) {
        if (!desc_ok(&t[i])) return ORC_E_INVALID;
        np += t[i].split == ORC_RESIDUAL_QKV ? 3 : 1;
    }
    L->parts = (part_t*)calloc(np, sizeof(part_t));
    if (!L->parts) return ORC_E_NOMEM;
    uint64_t k = 0, chunks = 0;
    for (uint32_t i = 0; i < n; ++i) {
        const orc_tensor* d = &t[i];
        int nsub = d->split == ORC_RESIDUAL_QKV ? 3 : 1;
        uint64_t roff = d->recv_off;
        for (int s = 0; s < nsub; ++s) {
            part_t* p = &L->parts[k++];
            p->desc = i;
            p->sub = (uint32_t)s;
            p->bits = d->elem_bits;
            p->cols = d->cols;
            if (d->split == ORC_RESIDUAL_QKV) {
                p->residual = 1;
                p->rows = (uint64_t)(s == 0 ? d->q_heads : d->kv_heads) * d->head_dim;
            } else {
                p->rows = d->rows;
            }
            p->bytes = p->rows * p->cols * p->bits / 8;
            p->recv_off = roff;
            roff += p->bytes;
            p->chunk0 = chunks;
            p->nchunks = (p->bytes + ORC_CHUNK - 1) / ORC_CHUNK;
            chunks += p->nchunks;
            L->canonical_bytes += p->bytes;
        }
    }
    L->n_parts = np;
    L->n_chunks = chunks;
    L->chunk_part = (uint64_t*)malloc(chunks * sizeof(uint64_t));
    L->win_start = (uint64_t*)malloc((chunks + 2) * sizeof(uint64_t));
    if (!L->chunk_part || !L->win_start) { layout_free(L); return ORC_E_NOMEM; }
    for (uint64_t p = 0; p < np; ++p)
        for (uint64_t c = 0; c < L->parts[p].nchunks; ++c) L->chunk_part[L->parts[p].chunk0 + c] = p;

    uint64_t nw = 0, cur = 0;
    L->win_start[nw++] = 0;
    uint64_t p = 0;
    for (uint32_t i = 0; i < n; ++i) {
        uint64_t p_end = p, B = 0;
        while (p_end < np && L->parts[p_end].desc == i) B += L->parts[p_end++].bytes;
        if (cur > 0 && cur + B > window_bytes) {
            L->win_start[nw++] = L->parts[p].chunk0;
            cur = 0;
        }
        for (; p < p_end; ++p) {
            for (uint64_t c = 0; c < L->parts[p].nchunks; ++c) {
                uint64_t len = L->parts[p].bytes - c * ORC_CHUNK;
                if (len > ORC_CHUNK) len = ORC_CHUNK;
                if (cur > 0 && cur + len > window_bytes) {
                    L->win_start[nw++] = L->parts[p].chunk0 + c;
                    cur = 0;
                }
                cur += len;
            }
        }
    }
    L->win_start[nw] = chunks;
    L->n_windows = nw;

    uint64_t h = 0xCBF29CE484222325ULL;
    fnv(&h, "DCR1", 4);
    fnv32(&h, ORC_CHUNK);
    fnv64(&h, window_bytes);
    fnv32(&h, (uint32_t)np);
    for (uint64_t q = 0; q < np; ++q) {
        fnv32(&h, L->parts[q].bits);
        fnv64(&h, L->parts[q].rows);
        fnv64(&h, L->parts[q].cols);
        fnv32(&h, L->parts[q].residual);
        fnv32(&h, L->parts[q].desc);
    }
    L->hash = h;
    return ORC_OK;
}

int orc_info_get(const orc_tensor* t, uint32_t n, uint64_t window_bytes, orc_info* out)
{
    layout_t L;
    int rc = layout_build(t, n, window_bytes, &L);
    if (rc) return rc;
    out->n_parts = L.n_parts;
    out->n_chunks = L.n_chunks;
    out->n_windows = L.n_windows;
    out->canonical_bytes = L.canonical_bytes;
    out->plan_hash = L.hash;
    layout_free(&L);
    return ORC_OK;
}

int orc_window_range(const orc_tensor* t, uint32_t n, uint64_t window_bytes, uint32_t w,
                     uint64_t* chunk_begin, uint64_t* chunk_count)
{
    layout_t L;
    int rc = layout_build(t, n, window_bytes, &L);
    if (rc) return rc;
    if (w >= L.n_windows) { layout_free(&L); return ORC_E_INVALID; }
    *chunk_begin = L.win_start[w];
    *chunk_count = L.win_start[w + 1] - L.win_start[w];
    layout_free(&L);
    return ORC_OK;
}

int orc_chunk_info(const orc_tensor* t, uint32_t n, uint64_t chunk, uint32_t* part_desc,
                   uint32_t* part_sub, uint64_t* part_off, uint32_t* len)
{
    layout_t L;
    int rc = layout_build(t, n, 1ULL << 62, &L);
    if (rc) return rc;
    if (chunk >= L.n_chunks) { layout_free(&L); return ORC_E_INVALID; }
    const part_t* p = &L.parts[L.chunk_part[chunk]];
    uint64_t off = (chunk - p->chunk0) * ORC_CHUNK;
    *part_desc = p->desc;
    *part_sub = p->sub;
    *part_off = off;
    *len = (uint32_t)((p->bytes - off) < ORC_CHUNK ? (p->bytes - off) : ORC_CHUNK);
    layout_free(&L);
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* element access (stored bits only; no arithmetic on values)               */
/* ------------------------------------------------------------------------ */
static inline uint32_t get_elem(const uint8_t* b, uint64_t i, uint32_t bits)
{
    if (bits == 16) return (uint32_t)b[2 * i] | ((uint32_t)b[2 * i + 1] << 8);
    if (bits == 8) return b[i];
    return (i & 1) ? (uint32_t)(b[i >> 1] >> 4) : (uint32_t)(b[i >> 1] & 15u);
}

static inline void set_elem(uint8_t* b, uint64_t i, uint32_t bits, uint32_t v)
{
    if (bits == 16) {
        b[2 * i] = (uint8_t)v;
        b[2 * i + 1] = (uint8_t)(v >> 8);
    } else if (bits == 8) {
        b[i] = (uint8_t)v;
    } else if (i & 1) {
        b[i >> 1] = (uint8_t)((b[i >> 1] & 0x0Fu) | ((v & 15u) << 4));
    } else {
        b[i >> 1] = (uint8_t)((b[i >> 1] & 0xF0u) | (v & 15u));
    }
}

/* Direct projection ([P1] "Direct Projection"; [P2] canonical coordinates):
 * canonical element (i, j) of a part -> (owner shard, local element index),
 * from the static shard layout alone.  Column-parallel tensors split dim 0,
 * row-parallel ones dim 1, replicated ones are owned by shard 0 ([P2] shard
 * owners).  The fused QKV of shard r holds kv groups g in
 * [r*G/tp, (r+1)*G/tp), each laid out as [its q heads | its k head | its v
 * head] ([P1] "Residual Conversion"; [P2] fused Q/K/V). */
static void src_of(const orc_tensor* d, uint32_t sub, uint64_t i, uint64_t j, uint32_t* r,
                   uint64_t* local)
{
    switch (d->split) {
    case ORC_REPLICATED:
        *r = 0;
        *local = i * d->cols + j;
        return;
    case ORC_SPLIT_ROWS: {
        uint64_t rl = d->rows / d->tp;
        *r = (uint32_t)(i / rl);
        *local = (i % rl) * d->cols + j;
        return;
    }
    case ORC_SPLIT_COLS: {
        uint64_t cl = d->cols / d->tp;
        *r = (uint32_t)(j / cl);
        *local = i * cl + (j % cl);
        return;
    }
    default: {
        uint64_t D = d->head_dim, G = d->kv_heads, qpg = d->q_heads / G, gpl = G / d->tp;
        uint64_t g, row_in_group;
        if (sub == 0) {
            uint64_t h = i / D;
            g = h / qpg;
            row_in_group = (h % qpg) * D + i % D;
        } else {
            g = i / D;
            row_in_group = (qpg + (sub - 1)) * D + i % D;
        }
        *r = (uint32_t)(g / gpl);
        *local = ((g % gpl) * (qpg + 2) * D + row_in_group) * d->cols + j;
        return;
    }
    }
}

/* Receiver placement: canonical element (i, j) -> element index in the
 * receiver arena.  The row-group layout pairs gate (slot 0) and up (slot 1)
 * rows in groups of g ([P4] "Working with low-precision RL"): physical row
 * (i / g) * 2g + slot * g + i % g of the fused tensor. */
static uint64_t recv_of(const orc_tensor* d, const part_t* p, uint64_t i, uint64_t j)
{
    uint64_t base = p->recv_off * 8 / p->bits;
    uint64_t row = i;
    if (d->recv_layout == ORC_RECV_ROWGROUP) {
        uint64_t g = d->recv_group;
        row = (i / g) * 2 * g + d->recv_slot * g + i % g;
    }
    return base + row * p->cols + j;
}

/* canonical bytes [off, off + len) of part p, gathered element by element */
static void canon_range(const orc_tensor* d, const part_t* p, const uint8_t* const* shards,
                        uint64_t off, uint64_t len, uint8_t* out)
{
    uint64_t e0 = off * 8 / p->bits, e1 = (off + len) * 8 / p->bits;
    for (uint64_t e = e0; e < e1; ++e) {
        uint64_t i = e / p->cols, j = e % p->cols;
        uint32_t r;
        uint64_t loc;
        src_of(d, p->sub, i, j, &r, &loc);
        set_elem(out, e - e0, p->bits, get_elem(shards[r] + d->shard_off[r], loc, p->bits));
    }
}

int orc_canonical(const orc_tensor* t, uint32_t sub, const uint8_t* const* shards, uint8_t* out)
{
    layout_t L;
    int rc = layout_build(t, 1, 1ULL << 62, &L);
    if (rc) return rc;
    if (sub >= L.n_parts) { layout_free(&L); return ORC_E_INVALID; }
    canon_range(t, &L.parts[sub], shards, 0, L.parts[sub].bytes, out);
    layout_free(&L);
    return ORC_OK;
}

/* Dense refit: every canonical element copied into its receiver place (the
 * full-checkpoint transfer the delta refit replaces; used to set up tests). */
int orc_receiver_dense(const orc_tensor* t, uint32_t n, const uint8_t* const* shards,
                       uint8_t* target)
{
    layout_t L;
    int rc = layout_build(t, n, 1ULL << 62, &L);
    if (rc) return rc;
    for (uint64_t q = 0; q < L.n_parts; ++q) {
        const part_t* p = &L.parts[q];
        const orc_tensor* d = &t[p->desc];
        for (uint64_t i = 0; i < p->rows; ++i)
            for (uint64_t j = 0; j < p->cols; ++j) {
                uint32_t r;
                uint64_t loc;
                src_of(d, p->sub, i, j, &r, &loc);
                set_elem(target, recv_of(d, p, i, j), p->bits,
                         get_elem(shards[r] + d->shard_off[r], loc, p->bits));
            }
    }
    layout_free(&L);
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* primitives                                                               */
/* ------------------------------------------------------------------------ */

/* [P4] "Delta update algebra": mask = weights_old XOR weights_new over the
 * raw bits, with no floating-point operation. */
void orc_xor(const uint8_t* a, const uint8_t* b, uint8_t* out, uint64_t n)
{
    for (uint64_t i = 0; i < n; ++i) out[i] = (uint8_t)(a[i] ^ b[i]);
}

/* [P1] change detection; [P2] shard owners: a stored value changed iff its
 * stored bits differ (so +0 vs -0 is a change).  Elements are 16-bit words,
 * bytes, or nibbles (low nibble first). */
uint64_t orc_count_changed(const uint8_t* mask, uint64_t nbytes, uint32_t elem_bits)
{
    uint64_t n = nbytes * 8 / elem_bits, c = 0;
    for (uint64_t e = 0; e < n; ++e) c += get_elem(mask, e, elem_bits) != 0;
    return c;
}

/* ---- LZ4 block format ([P4] footnote 4 names the LZ4 block format) -------
 * A block is a series of sequences: a token (high nibble literal length, low
 * nibble match length - 4, 15 meaning "more length bytes follow, each 255
 * continuing"), the literal bytes, a 2-byte little-endian offset, then the
 * optional match-length bytes.  The last sequence holds literals only.
 * Minimum match 4; the encoder keeps the last 5 bytes as literals and starts
 * no match in the last 12 bytes. */
#define LZ4_MINMATCH 4u
#define LZ4_LASTLITERALS 5u
#define LZ4_MFLIMIT 12u
#define LZ4_HASHLOG 14u

static inline uint32_t rd32(const uint8_t* p)
{
    return (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) | ((uint32_t)p[3] << 24);
}

static uint64_t put_len(uint8_t* out, uint64_t o, uint64_t cap, uint64_t v, int* ovf)
{
    /* v >= 15 already stored as 15 in the token; emit v - 15 in 255-steps */
    v -= 15;
    while (v >= 255) {
        if (o >= cap) { *ovf = 1; return o; }
        out[o++] = 255;
        v -= 255;
    }
    if (o >= cap) { *ovf = 1; return o; }
    out[o++] = (uint8_t)v;
    return o;
}

static uint64_t put_seq(uint8_t* out, uint64_t o, uint64_t cap, const uint8_t* lit, uint64_t ll,
                        uint32_t off, uint64_t ml, int last, int* ovf)
{
    uint64_t mcode = last ? 0 : ml - LZ4_MINMATCH;
    if (o >= cap) { *ovf = 1; return o; }
    out[o++] = (uint8_t)(((ll >= 15 ? 15 : ll) << 4) | (mcode >= 15 ? 15 : mcode));
    if (ll >= 15) o = put_len(out, o, cap, ll, ovf);
    if (*ovf || o + ll > cap) { *ovf = 1; return o; }
    memcpy(out + o, lit, ll);
    o += ll;
    if (last) return o;
    if (o + 2 > cap) { *ovf = 1; return o; }
    out[o++] = (uint8_t)off;
    out[o++] = (uint8_t)(off >> 8);
    if (mcode >= 15) o = put_len(out, o, cap, mcode, ovf);
    return o;
}

/* Plain greedy encoder: a 2^14-entry table of the most recent position of
 * each 4-byte word's Knuth multiplicative hash; every position is inserted
 * (match interiors included); a candidate is taken when its 4 bytes are equal
 * and it lies within 65535 bytes; matches extend forward only, no lazy
 * evaluation.  Returns the block size, or 0 if cap is too small. */
uint64_t orc_lz4_encode(const uint8_t* in, uint64_t n, uint8_t* out, uint64_t cap)
{
    int32_t* tab = (int32_t*)malloc(sizeof(int32_t) << LZ4_HASHLOG);
    if (!tab) return 0;
    for (uint32_t i = 0; i < (1u << LZ4_HASHLOG); ++i) tab[i] = -1;
    int ovf = 0;
    uint64_t o = 0, anchor = 0, p = 0;
    while (n >= LZ4_MFLIMIT && p <= n - LZ4_MFLIMIT) {
        uint32_t w = rd32(in + p);
        uint32_t h = (uint32_t)(w * 2654435761u) >> (32 - LZ4_HASHLOG);
        int32_t cand = tab[h];
        tab[h] = (int32_t)p;
        if (cand >= 0 && p - (uint64_t)cand <= 65535 && rd32(in + cand) == w) {
            uint64_t len = LZ4_MINMATCH;
            while (p + len < n - LZ4_LASTLITERALS && in[cand + len] == in[p + len]) ++len;
            o = put_seq(out, o, cap, in + anchor, p - anchor, (uint32_t)(p - (uint64_t)cand), len, 0,
                        &ovf);
            if (ovf) break;
            for (uint64_t q = p + 1; q < p + len && q + 4 <= n; ++q) {
                uint32_t wq = rd32(in + q);
                tab[(uint32_t)(wq * 2654435761u) >> (32 - LZ4_HASHLOG)] = (int32_t)q;
            }
            p += len;
            anchor = p;
        } else {
            ++p;
        }
    }
    if (!ovf) o = put_seq(out, o, cap, in + anchor, n - anchor, 0, 0, 1, &ovf);
    free(tab);
    return ovf ? 0 : o;
}

/* Strict decoder: accepts any block whose every read and write stays in
 * bounds and that yields exactly raw_len bytes; rejects offset 0, offsets
 * beyond the bytes produced so far, truncation and overruns.  Overlapping
 * copies replicate forward byte by byte.  With zsrc set, every match must
 * copy only zero bytes (frames that promise this carry the ZSRC flag). */
int orc_lz4_decode(const uint8_t* in, uint64_t n, uint8_t* out, uint64_t raw_len, uint32_t zsrc)
{
    uint64_t ip = 0, op = 0;
    for (;;) {
        if (ip >= n) return ORC_E_CORRUPT;
        uint32_t tok = in[ip++];
        uint64_t ll = tok >> 4;
        if (ll == 15) {
            for (;;) {
                if (ip >= n) return ORC_E_CORRUPT;
                uint32_t b = in[ip++];
                ll += b;
                if (b != 255) break;
            }
        }
        if (ll > n - ip || ll > raw_len - op) return ORC_E_CORRUPT;
        memcpy(out + op, in + ip, ll);
        ip += ll;
        op += ll;
        if (ip == n) break;
        if (n - ip < 2) return ORC_E_CORRUPT;
        uint64_t off = (uint64_t)in[ip] | ((uint64_t)in[ip + 1] << 8);
        ip += 2;
        if (off == 0 || off > op) return ORC_E_CORRUPT;
        uint64_t ml = tok & 15u;
        if (ml == 15) {
            for (;;) {
                if (ip >= n) return ORC_E_CORRUPT;
                uint32_t b = in[ip++];
                ml += b;
                if (b != 255) break;
            }
        }
        ml += LZ4_MINMATCH;
        if (ml > raw_len - op) return ORC_E_CORRUPT;
        for (uint64_t k = 0; k < ml; ++k) {
            uint8_t v = out[op + k - off];
            if (zsrc && v) return ORC_E_CORRUPT;
            out[op + k] = v;
        }
        op += ml;
    }
    return op == raw_len ? ORC_OK : ORC_E_CORRUPT;
}

/* ---- Snappy block format ([P4] "A strong baseline with the Blackwell-
 * native DE", footnote 4: LZ4 and Snappy are byte-oriented LZ77 codecs with
 * literals and back copies and no entropy stage; one Snappy copy covers at
 * most 64 bytes).  A block is the uncompressed length as a little-endian
 * base-128 varint, then elements whose tag byte's low two bits give the type:
 *   0 literal: length - 1 in the upper six bits when below 60; 60..63 mean
 *     that 1..4 following bytes (little-endian) hold length - 1;
 *   1 copy: length 4..11 as length - 4 in bits 2..4, offset bits 8..10 in
 *     bits 5..7, then the offset's low byte;
 *   2 copy: length 1..64 as length - 1 in the upper six bits, then a 2-byte
 *     little-endian offset;
 *   3 copy: the same with a 4-byte offset.
 * Copies replicate forward byte by byte when they overlap. */
static uint64_t sn_literal(uint8_t* out, uint64_t o, uint64_t cap, const uint8_t* lit, uint64_t ll, int* ovf)
{
    if (ll == 0) return o;
    uint64_t v = ll - 1, nb = v < 60 ? 0 : v < 256 ? 1 : v < 65536 ? 2 : v < (1ull << 24) ? 3 : 4;
    if (o + 1 + nb + ll > cap) { *ovf = 1; return o; }
    out[o++] = (uint8_t)((nb ? 59 + nb : v) << 2);
    for (uint64_t i = 0; i < nb; ++i) out[o++] = (uint8_t)(v >> (8 * i));
    memcpy(out + o, lit, ll);
    return o + ll;
}

static uint64_t sn_copy(uint8_t* out, uint64_t o, uint64_t cap, uint64_t off, uint64_t len, int* ovf)
{
    if (len >= 4 && len <= 11 && off < 2048) {
        if (o + 2 > cap) { *ovf = 1; return o; }
        out[o++] = (uint8_t)(1 | ((len - 4) << 2) | ((off >> 8) << 5));
        out[o++] = (uint8_t)off;
    } else {
        if (o + 3 > cap) { *ovf = 1; return o; }
        out[o++] = (uint8_t)(2 | ((len - 1) << 2));
        out[o++] = (uint8_t)off;
        out[o++] = (uint8_t)(off >> 8);
    }
    return o;
}

/* a match of len >= 4 bytes as copies of at most 64: 64 while at least 68
 * remain, 60 if more than 64 remain, then the rest (never below 4) */
static uint64_t sn_match(uint8_t* out, uint64_t o, uint64_t cap, uint64_t off, uint64_t len, int* ovf)
{
    while (len >= 68 && !*ovf) {
        o = sn_copy(out, o, cap, off, 64, ovf);
        len -= 64;
    }
    if (len > 64 && !*ovf) {
        o = sn_copy(out, o, cap, off, 60, ovf);
        len -= 60;
    }
    if (!*ovf) o = sn_copy(out, o, cap, off, len, ovf);
    return o;
}

/* Plain greedy encoder with the same match finder as orc_lz4_encode (2^14
 * slots of the most recent position of each 4-byte word's hash, every
 * position inserted, forward extension only, offsets up to 65535); the
 * format has no end-of-block rules, so matches may reach the last byte.
 * Returns the block size, or 0 if cap is too small. */
uint64_t orc_snappy_encode(const uint8_t* in, uint64_t n, uint8_t* out, uint64_t cap)
{
    int32_t* tab = (int32_t*)malloc(sizeof(int32_t) << LZ4_HASHLOG);
    if (!tab) return 0;
    for (uint32_t i = 0; i < (1u << LZ4_HASHLOG); ++i) tab[i] = -1;
    int ovf = 0;
    uint64_t o = 0, anchor = 0, p = 0;
    for (uint64_t v = n;; v >>= 7) {   /* preamble */
        if (o >= cap) { ovf = 1; break; }
        out[o++] = (uint8_t)((v & 127) | (v >= 128 ? 128 : 0));
        if (v < 128) break;
    }
    while (!ovf && p + 4 <= n) {
        uint32_t w = rd32(in + p);
        uint32_t h = (uint32_t)(w * 2654435761u) >> (32 - LZ4_HASHLOG);
        int32_t cand = tab[h];
        tab[h] = (int32_t)p;
        if (cand >= 0 && p - (uint64_t)cand <= 65535 && rd32(in + cand) == w) {
            uint64_t len = 4;
            while (p + len < n && in[cand + len] == in[p + len]) ++len;
            o = sn_literal(out, o, cap, in + anchor, p - anchor, &ovf);
            if (!ovf) o = sn_match(out, o, cap, p - (uint64_t)cand, len, &ovf);
            for (uint64_t q = p + 1; q < p + len && q + 4 <= n; ++q) {
                uint32_t wq = rd32(in + q);
                tab[(uint32_t)(wq * 2654435761u) >> (32 - LZ4_HASHLOG)] = (int32_t)q;
            }
            p += len;
            anchor = p;
        } else {
            ++p;
        }
    }
    if (!ovf) o = sn_literal(out, o, cap, in + anchor, n - anchor, &ovf);
    free(tab);
    return ovf ? 0 : o;
}

/* Strict decoder: the preamble must equal raw_len and fit in five bytes;
 * every element must stay inside the block and the output; offsets must be
 * non-zero and within the bytes produced so far; the block must produce
 * exactly raw_len bytes.  With zsrc set, every copy must copy zero bytes. */
int orc_snappy_decode(const uint8_t* in, uint64_t n, uint8_t* out, uint64_t raw_len, uint32_t zsrc)
{
    uint64_t ip = 0, op = 0, v = 0;
    for (uint32_t shift = 0;; shift += 7) {
        if (ip >= n || shift > 28) return ORC_E_CORRUPT;
        uint32_t b = in[ip++];
        v |= (uint64_t)(b & 127) << shift;
        if (!(b & 128)) break;
    }
    if (v != raw_len) return ORC_E_CORRUPT;
    while (ip < n) {
        uint32_t tag = in[ip++];
        uint64_t len, off;
        if ((tag & 3) == 0) {
            len = (uint64_t)(tag >> 2) + 1;
            if ((tag >> 2) >= 60) {
                uint32_t nb = (tag >> 2) - 59;
                if (nb > n - ip) return ORC_E_CORRUPT;
                len = 0;
                for (uint32_t i = 0; i < nb; ++i) len |= (uint64_t)in[ip + i] << (8 * i);
                len += 1;
                ip += nb;
            }
            if (len > n - ip || len > raw_len - op) return ORC_E_CORRUPT;
            memcpy(out + op, in + ip, len);
            ip += len;
            op += len;
            continue;
        }
        if ((tag & 3) == 1) {
            if (ip >= n) return ORC_E_CORRUPT;
            len = ((tag >> 2) & 7) + 4;
            off = ((uint64_t)(tag >> 5) << 8) | in[ip++];
        } else {
            uint32_t nb = (tag & 3) == 2 ? 2 : 4;
            if (nb > n - ip) return ORC_E_CORRUPT;
            len = (uint64_t)(tag >> 2) + 1;
            off = 0;
            for (uint32_t i = 0; i < nb; ++i) off |= (uint64_t)in[ip + i] << (8 * i);
            ip += nb;
        }
        if (off == 0 || off > op || len > raw_len - op) return ORC_E_CORRUPT;
        for (uint64_t k = 0; k < len; ++k) {
            uint8_t b = out[op + k - off];
            if (zsrc && b) return ORC_E_CORRUPT;
            out[op + k] = b;
        }
        op += len;
    }
    return op == raw_len ? ORC_OK : ORC_E_CORRUPT;
}

/* ------------------------------------------------------------------------ */
/* stream encode                                                            */
/* ------------------------------------------------------------------------ */
static void put32(uint8_t* p, uint32_t v)
{
    p[0] = (uint8_t)v; p[1] = (uint8_t)(v >> 8); p[2] = (uint8_t)(v >> 16); p[3] = (uint8_t)(v >> 24);
}
static void put64(uint8_t* p, uint64_t v)
{
    put32(p, (uint32_t)v);
    put32(p + 4, (uint32_t)(v >> 32));
}
static uint32_t get32(const uint8_t* p) { return rd32(p); }
static uint64_t get64(const uint8_t* p) { return (uint64_t)rd32(p) | ((uint64_t)rd32(p + 4) << 32); }

#define STREAM_HDR 64u
#define FRAME_HDR 32u
#define STREAM_MAGIC 0x53524344u /* "DCRS" */
#define FRAME_MAGIC 0x46524344u  /* "DCRF" */
#define FLAG_OVERWRITE_ONLY 1u
#define FRAME_ZSRC 1u

typedef struct {
    const orc_tensor* t;
    const layout_t* L;
    const uint8_t* const* olds;
    const uint8_t* const* news;
    uint32_t mode;
    uint32_t codec;
    uint64_t cb, cc;
    uint8_t** frames;
    uint64_t* flen;
    uint64_t* changed;
    atomic_ullong next;
    atomic_int err;
} enc_job;

/* One chunk: canonicalise old and new ([P1] direct projection / residual
 * conversion), mask and count ([P4] delta algebra; [P2] bitwise compare),
 * then encode ([P1] hybrid encoding: XOR masks LZ4-compressed for affine
 * changes, overwrites for residual ones; [P3] same split). */
static int encode_chunk(enc_job* J, uint64_t c, uint8_t* old_c, uint8_t* new_c, uint8_t* mask,
                        uint8_t* tmp, uint64_t tmp_cap)
{
    const part_t* p = &J->L->parts[J->L->chunk_part[c]];
    const orc_tensor* d = &J->t[p->desc];
    uint64_t off = (c - p->chunk0) * ORC_CHUNK;
    uint64_t len = p->bytes - off < ORC_CHUNK ? p->bytes - off : ORC_CHUNK;
    canon_range(d, p, J->olds, off, len, old_c);
    canon_range(d, p, J->news, off, len, new_c);
    orc_xor(old_c, new_c, mask, len);
    uint64_t changed = orc_count_changed(mask, len, p->bits);
    uint64_t k = c - J->cb;
    J->changed[k] = changed;
    J->frames[k] = NULL;
    J->flen[k] = 0;
    if (changed == 0) return ORC_OK;

    uint32_t kind;
    uint64_t body_len;
    const uint8_t* body;
    if (p->residual || J->mode == ORC_MODE_OVERWRITE_ONLY) {
        uint32_t ub = p->bits == 16 ? 2 : 1;
        uint64_t nu = len / ub, cnt = 0;
        for (uint64_t u = 0; u < nu; ++u) {
            int ch = 0;
            for (uint32_t b = 0; b < ub; ++b) ch |= mask[u * ub + b] != 0;
            cnt += ch;
        }
        uint64_t pad = (4 - (2 * cnt) % 4) % 4;
        uint64_t rec = 4 + 2 * cnt + pad + cnt * ub;
        if (rec >= len) {
            kind = ORC_K_OVERWRITE_DENSE;
            body = new_c;
            body_len = len;
        } else {
            kind = ORC_K_OVERWRITE;
            put32(tmp, (uint32_t)cnt);
            uint64_t o = 4, v = 4 + 2 * cnt + pad;
            memset(tmp + 4 + 2 * cnt, 0, pad);
            for (uint64_t u = 0; u < nu; ++u) {
                int ch = 0;
                for (uint32_t b = 0; b < ub; ++b) ch |= mask[u * ub + b] != 0;
                if (!ch) continue;
                tmp[o++] = (uint8_t)u;
                tmp[o++] = (uint8_t)(u >> 8);
                for (uint32_t b = 0; b < ub; ++b) tmp[v++] = new_c[u * ub + b];
            }
            body = tmp;
            body_len = rec;
        }
    } else {
        const int sn = J->codec == ORC_CODEC_SNAPPY;
        uint64_t lz = sn ? orc_snappy_encode(mask, len, tmp, tmp_cap) : orc_lz4_encode(mask, len, tmp, tmp_cap);
        if (lz == 0 || lz >= len) {
            kind = ORC_K_XOR_RAW;
            body = mask;
            body_len = len;
        } else {
            kind = sn ? ORC_K_XOR_SNAPPY : ORC_K_XOR_LZ4;
            body = tmp;
            body_len = lz;
        }
    }
    uint64_t fl = (FRAME_HDR + body_len + 15) / 16 * 16;
    uint8_t* f = (uint8_t*)calloc(fl, 1);
    if (!f) return ORC_E_NOMEM;
    put32(f, FRAME_MAGIC);
    f[4] = (uint8_t)kind;
    f[5] = (uint8_t)p->bits;
    f[6] = 0;
    f[7] = 0;
    put32(f + 8, (uint32_t)c);
    put32(f + 12, (uint32_t)len);
    put32(f + 16, (uint32_t)body_len);
    put32(f + 20, (uint32_t)changed);
    memcpy(f + FRAME_HDR, body, body_len);
    J->frames[k] = f;
    J->flen[k] = fl;
    return ORC_OK;
}

static void* enc_worker(void* arg)
{
    enc_job* J = (enc_job*)arg;
    uint64_t tmp_cap = ORC_CHUNK * 2 + 64;
    uint8_t* buf = (uint8_t*)malloc(ORC_CHUNK * 3 + tmp_cap);
    if (!buf) { atomic_store(&J->err, ORC_E_NOMEM); return NULL; }
    for (;;) {
        uint64_t k = atomic_fetch_add(&J->next, 1);
        if (k >= J->cc) break;
        int rc = encode_chunk(J, J->cb + k, buf, buf + ORC_CHUNK, buf + 2 * ORC_CHUNK,
                              buf + 3 * ORC_CHUNK, tmp_cap);
        if (rc) { atomic_store(&J->err, rc); break; }
    }
    free(buf);
    return NULL;
}

static void run_pool(void* (*fn)(void*), void* arg, uint32_t threads)
{
    if (threads <= 1) { fn(arg); return; }
    pthread_t* th = (pthread_t*)malloc(threads * sizeof(pthread_t));
    uint32_t started = 0;
    for (uint32_t i = 0; th && i < threads; ++i)
        if (pthread_create(&th[i], NULL, fn, arg) == 0) ++started;
    if (started == 0) fn(arg);
    for (uint32_t i = 0; i < started; ++i) pthread_join(th[i], NULL);
    free(th);
}

/* Stream: 64-byte header, frames in ascending chunk order (each 16-byte
 * aligned, 32-byte frame header), then an index of the frames' offsets.
 * A chunk whose mask is all zero sends no frame. */
int orc_encode(const orc_tensor* t, uint32_t n, uint64_t window_bytes,
               const uint8_t* const* old_shards, const uint8_t* const* new_shards,
               uint32_t mode, uint32_t codec, uint32_t window, uint64_t base_version,
               uint64_t target_version, uint32_t threads, uint8_t* out, uint64_t cap, uint64_t* size,
               uint64_t* changed_per_tensor)
{
    if (!old_shards || !new_shards || !size || mode > ORC_MODE_OVERWRITE_ONLY || codec > ORC_CODEC_SNAPPY)
        return ORC_E_INVALID;
    layout_t L;
    int rc = layout_build(t, n, window_bytes, &L);
    if (rc) return rc;
    if (window >= L.n_windows) { layout_free(&L); return ORC_E_INVALID; }
    enc_job J;
    memset(&J, 0, sizeof(J));
    J.t = t;
    J.L = &L;
    J.olds = old_shards;
    J.news = new_shards;
    J.mode = mode;
    J.codec = codec;
    J.cb = L.win_start[window];
    J.cc = L.win_start[window + 1] - J.cb;
    J.frames = (uint8_t**)calloc(J.cc + 1, sizeof(uint8_t*));
    J.flen = (uint64_t*)calloc(J.cc + 1, sizeof(uint64_t));
    J.changed = (uint64_t*)calloc(J.cc + 1, sizeof(uint64_t));
    atomic_init(&J.next, 0);
    atomic_init(&J.err, 0);
    if (!J.frames || !J.flen || !J.changed) rc = ORC_E_NOMEM;
    if (!rc) {
        run_pool(enc_worker, &J, threads ? threads : 1);
        rc = atomic_load(&J.err);
    }
    if (!rc) {
        uint64_t nf = 0, fb = 0;
        for (uint64_t k = 0; k < J.cc; ++k)
            if (J.frames[k]) { ++nf; fb += J.flen[k]; }
        uint64_t total = STREAM_HDR + fb + 8 * nf;
        *size = total;
        if (changed_per_tensor) {
            for (uint32_t i = 0; i < n; ++i) changed_per_tensor[i] = 0;
            for (uint64_t k = 0; k < J.cc; ++k)
                changed_per_tensor[L.parts[L.chunk_part[J.cb + k]].desc] += J.changed[k];
        }
        if (!out || total > cap) {
            rc = ORC_E_CAPACITY;
        } else {
            memset(out, 0, STREAM_HDR);
            put32(out, STREAM_MAGIC);
            put32(out + 4, 1);
            put64(out + 8, L.hash);
            put64(out + 16, base_version);
            put64(out + 24, target_version);
            put32(out + 32, window);
            put32(out + 36, mode == ORC_MODE_OVERWRITE_ONLY ? FLAG_OVERWRITE_ONLY : 0);
            put32(out + 40, (uint32_t)J.cb);
            put32(out + 44, (uint32_t)J.cc);
            put64(out + 48, nf);
            put64(out + 56, total);
            uint64_t o = STREAM_HDR, idx = STREAM_HDR + fb;
            for (uint64_t k = 0; k < J.cc; ++k) {
                if (!J.frames[k]) continue;
                memcpy(out + o, J.frames[k], J.flen[k]);
                put64(out + idx, o);
                idx += 8;
                o += J.flen[k];
            }
        }
    }
    for (uint64_t k = 0; J.frames && k < J.cc; ++k) free(J.frames[k]);
    free(J.frames);
    free(J.flen);
    free(J.changed);
    layout_free(&L);
    return rc;
}

/* ------------------------------------------------------------------------ */
/* receiver                                                                 */
/* ------------------------------------------------------------------------ */
/* Receiver state ([P1] recoverable in-place apply, joint commit; [P2] dedup
 * by unique IDs): the committed version and, per chunk, the version it was
 * last claimed for with NOT_STARTED / CLAIMED / DONE.  The dedup ID of a
 * frame is (target_version, chunk_id). */
struct orc_state {
    uint64_t version, pending, n_chunks, n_windows;
    uint8_t* win_done;
    _Atomic uint64_t* chunk;   /* (version << 2) | state */
};
enum { ST_NOT_STARTED = 0, ST_CLAIMED = 1, ST_DONE = 2 };

orc_state* orc_state_new(const orc_tensor* t, uint32_t n, uint64_t window_bytes, uint64_t version)
{
    layout_t L;
    if (layout_build(t, n, window_bytes, &L)) return NULL;
    orc_state* s = (orc_state*)calloc(1, sizeof(orc_state));
    if (s) {
        s->version = version;
        s->pending = ~0ULL;
        s->n_chunks = L.n_chunks;
        s->n_windows = L.n_windows;
        s->win_done = (uint8_t*)calloc(L.n_windows, 1);
        s->chunk = (_Atomic uint64_t*)calloc(L.n_chunks ? L.n_chunks : 1, sizeof(uint64_t));
        if (!s->win_done || !s->chunk) { orc_state_free(s); s = NULL; }
    }
    layout_free(&L);
    return s;
}

void orc_state_free(orc_state* s)
{
    if (!s) return;
    free(s->win_done);
    free((void*)s->chunk);
    free(s);
}

uint64_t orc_state_version(const orc_state* s) { return s ? s->version : 0; }

typedef struct {
    const orc_tensor* t;
    const layout_t* L;
    orc_state* s;
    const uint8_t* payload;
    uint64_t frames_end, nf, cb, cc, V;
    uint8_t* target;
    uint32_t retry_only, split, dedup;
    uint64_t abort_at;
    atomic_ullong next;
    atomic_int err;
    atomic_int aborted;
} app_job;

/* apply canonical chunk bytes [0, lim) of a mask (XOR) to the receiver */
static void apply_xor(const app_job* A, const part_t* p, uint64_t off, const uint8_t* mask,
                      uint64_t lim)
{
    const orc_tensor* d = &A->t[p->desc];
    uint64_t e0 = off * 8 / p->bits, n = lim * 8 / p->bits;
    for (uint64_t e = 0; e < n; ++e) {
        uint32_t m = get_elem(mask, e, p->bits);
        if (!m) continue;
        uint64_t ce = e0 + e;
        uint64_t r = recv_of(d, p, ce / p->cols, ce % p->cols);
        set_elem(A->target, r, p->bits, get_elem(A->target, r, p->bits) ^ m);
    }
}

/* overwrite canonical chunk bytes with the given new bytes (unit-wise) */
static void apply_put(const app_job* A, const part_t* p, uint64_t off, uint64_t byte_in_chunk,
                      const uint8_t* v, uint64_t nbytes)
{
    const orc_tensor* d = &A->t[p->desc];
    uint64_t epb = 8 / p->bits ? 8 / p->bits : 1; /* elements per byte (16-bit: 1 per 2 bytes) */
    if (p->bits == 16) {
        for (uint64_t b = 0; b < nbytes; b += 2) {
            uint64_t ce = (off + byte_in_chunk + b) / 2;
            uint64_t r = recv_of(d, p, ce / p->cols, ce % p->cols);
            set_elem(A->target, r, 16, (uint32_t)v[b] | ((uint32_t)v[b + 1] << 8));
        }
        return;
    }
    for (uint64_t b = 0; b < nbytes; ++b) {
        for (uint64_t k = 0; k < epb; ++k) {
            uint64_t ce = (off + byte_in_chunk + b) * epb + k;
            uint32_t val = p->bits == 8 ? v[b] : (k ? (uint32_t)(v[b] >> 4) : (uint32_t)(v[b] & 15u));
            uint64_t r = recv_of(d, p, ce / p->cols, ce % p->cols);
            set_elem(A->target, r, p->bits, val);
        }
    }
}

static int apply_frame(app_job* A, uint64_t f, uint8_t* mask)
{
    const uint8_t* pl = A->payload;
    uint64_t fo = get64(pl + A->frames_end + 8 * f);
    if (fo < STREAM_HDR || fo > A->frames_end || A->frames_end - fo < FRAME_HDR || fo % 16)
        return ORC_E_CORRUPT;
    const uint8_t* h = pl + fo;
    uint32_t kind = h[4], bits = h[5], flags = (uint32_t)h[6] | ((uint32_t)h[7] << 8);
    uint64_t c = get32(h + 8), raw = get32(h + 12), bl = get32(h + 16);
    if (get32(h) != FRAME_MAGIC || kind < ORC_K_XOR_LZ4 || kind > ORC_K_XOR_SNAPPY)
        return ORC_E_CORRUPT;
    if (c < A->cb || c >= A->cb + A->cc || bl > A->frames_end - fo - FRAME_HDR) return ORC_E_CORRUPT;
    const part_t* p = &A->L->parts[A->L->chunk_part[c]];
    uint64_t off = (c - p->chunk0) * ORC_CHUNK;
    uint64_t len = p->bytes - off < ORC_CHUNK ? p->bytes - off : ORC_CHUNK;
    if (raw != len || bits != p->bits) return ORC_E_CORRUPT;
    int is_xor = kind == ORC_K_XOR_LZ4 || kind == ORC_K_XOR_RAW || kind == ORC_K_XOR_SNAPPY;
    if (A->retry_only && is_xor) return ORC_E_INVALID;
    if (f > A->abort_at) return ORC_OK; /* injected fault: never reached */
    int cut = f == A->abort_at;
    uint64_t lim = cut ? (A->split < len ? A->split : len) : len;
    lim -= lim % (p->bits == 16 ? 2u : 1u);   /* a split falls on an element boundary */
    const uint8_t* body = h + FRAME_HDR;
    _Atomic uint64_t* st = &A->s->chunk[c];
    uint64_t claimed = (A->V << 2) | ST_CLAIMED, done = (A->V << 2) | ST_DONE;

    if (is_xor) {
        /* [P2] dedup: a mask is never applied twice to one chunk */
        if (A->dedup) {
            uint64_t cur = atomic_load(st);
            for (;;) {
                if ((cur >> 2) == A->V && (cur & 3) != ST_NOT_STARTED) return ORC_OK;
                if (atomic_compare_exchange_weak(st, &cur, claimed)) break;
            }
        }
        if (kind == ORC_K_XOR_RAW) {
            if (bl != raw) return ORC_E_CORRUPT;
            memcpy(mask, body, raw);
        } else if (kind == ORC_K_XOR_SNAPPY) {
            if (orc_snappy_decode(body, bl, mask, raw, flags & FRAME_ZSRC) != ORC_OK) return ORC_E_CORRUPT;
        } else if (orc_lz4_decode(body, bl, mask, raw, flags & FRAME_ZSRC) != ORC_OK) {
            return ORC_E_CORRUPT;
        }
        apply_xor(A, p, off, mask, lim);   /* [P1], [P2]: XOR in place, no backup */
    } else if (kind == ORC_K_OVERWRITE_DENSE) {
        if (bl != raw) return ORC_E_CORRUPT;
        apply_put(A, p, off, 0, body, lim);
    } else {
        /* [P1] overwrite records replace the stored values; idempotent ([P2]) */
        uint32_t ub = p->bits == 16 ? 2 : 1;
        if (bl < 4) return ORC_E_CORRUPT;
        uint64_t cnt = get32(body);
        uint64_t pad = (4 - (2 * cnt) % 4) % 4;
        if (4 + 2 * cnt + pad + cnt * ub != bl) return ORC_E_CORRUPT;
        const uint8_t* vals = body + 4 + 2 * cnt + pad;
        uint64_t prev = 0;
        for (uint64_t k = 0; k < cnt; ++k) {
            uint64_t u = (uint64_t)body[4 + 2 * k] | ((uint64_t)body[5 + 2 * k] << 8);
            if ((u + 1) * ub > raw || (k && u <= prev)) return ORC_E_CORRUPT;
            prev = u;
        }
        for (uint64_t k = 0; k < cnt; ++k) {
            uint64_t u = (uint64_t)body[4 + 2 * k] | ((uint64_t)body[5 + 2 * k] << 8);
            if (u * ub >= lim) continue;
            apply_put(A, p, off, u * ub, vals + k * ub, ub);
        }
    }
    if (cut) {
        atomic_store(&A->aborted, 1);
        if (!is_xor || !A->dedup) atomic_store(st, claimed);
    } else {
        atomic_store(st, done);
    }
    return ORC_OK;
}

static void* app_worker(void* arg)
{
    app_job* A = (app_job*)arg;
    uint8_t* mask = (uint8_t*)malloc(ORC_CHUNK);
    if (!mask) { atomic_store(&A->err, ORC_E_NOMEM); return NULL; }
    for (;;) {
        uint64_t f = atomic_fetch_add(&A->next, 1);
        if (f >= A->nf) break;
        int rc = apply_frame(A, f, mask);
        if (rc) {
            int z = 0;
            atomic_compare_exchange_strong(&A->err, &z, rc);
        }
    }
    free(mask);
    return NULL;
}

/* [P1] recoverable in-place apply and joint commit; [P2] in-place apply, dedup,
 * overwrite-only retry; [P3] retries overwrite partial writes and a joint
 * commit binds the new version as the next base. */
int orc_apply(const orc_tensor* t, uint32_t n, uint64_t window_bytes, orc_state* s,
              const uint8_t* payload, uint64_t size, uint8_t* target, uint32_t retry_only,
              uint64_t abort_at, uint32_t split, uint32_t dedup, uint32_t threads)
{
    if (!s || !payload || !target || size < STREAM_HDR) return ORC_E_INVALID;
    layout_t L;
    int rc = layout_build(t, n, window_bytes, &L);
    if (rc) return rc;
    const uint8_t* h = payload;
    uint64_t nf = get64(h + 48), total = get64(h + 56);
    uint32_t w = get32(h + 32), fl = get32(h + 36);
    if (get32(h) != STREAM_MAGIC || get32(h + 4) != 1 || total > size || total < STREAM_HDR ||
        nf > (total - STREAM_HDR) / 8) {
        rc = ORC_E_CORRUPT;
    } else if (get64(h + 8) != L.hash || w >= L.n_windows || L.n_chunks != s->n_chunks ||
               get32(h + 40) != L.win_start[w] ||
               get32(h + 44) != L.win_start[w + 1] - L.win_start[w]) {
        rc = ORC_E_INVALID;
    } else if (retry_only && !(fl & FLAG_OVERWRITE_ONLY)) {
        rc = ORC_E_INVALID;
    } else if (get64(h + 16) != s->version) {
        rc = ORC_E_VERSION;
    }
    if (rc) { layout_free(&L); return rc; }

    uint64_t V = get64(h + 24);
    if (V != s->pending) {
        memset(s->win_done, 0, s->n_windows);
        s->pending = V;
    }
    app_job A;
    memset(&A, 0, sizeof(A));
    A.t = t;
    A.L = &L;
    A.s = s;
    A.payload = payload;
    A.nf = nf;
    A.frames_end = total - 8 * nf;
    A.cb = L.win_start[w];
    A.cc = L.win_start[w + 1] - A.cb;
    A.V = V;
    A.target = target;
    A.retry_only = retry_only;
    A.split = split;
    A.dedup = dedup;
    A.abort_at = abort_at;
    atomic_init(&A.next, 0);
    atomic_init(&A.err, 0);
    atomic_init(&A.aborted, 0);
    run_pool(app_worker, &A, threads ? threads : 1);
    rc = atomic_load(&A.err);

    /* commit rule: every chunk with a frame in this stream is DONE for V */
    uint64_t pending = 0;
    for (uint64_t f = 0; f < nf; ++f) {
        uint64_t fo = get64(payload + A.frames_end + 8 * f);
        if (fo < STREAM_HDR || fo + FRAME_HDR > A.frames_end) { ++pending; continue; }
        uint64_t c = get32(payload + fo + 8);
        if (c < A.cb || c >= A.cb + A.cc) { ++pending; continue; }
        if (atomic_load(&s->chunk[c]) != ((V << 2) | ST_DONE)) ++pending;
    }
    if (!rc && atomic_load(&A.aborted)) rc = ORC_E_ABORTED;
    if (!rc && pending) rc = ORC_E_INCOMPLETE;
    if (!rc) {
        s->win_done[w] = 1;
        int all = 1;
        for (uint64_t k = 0; k < s->n_windows; ++k) all &= s->win_done[k];
        if (all) {
            s->version = V;
            s->pending = ~0ULL;
        }
    }
    layout_free(&L);
    return rc;
}
