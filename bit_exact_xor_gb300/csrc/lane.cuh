// One thread's walk of a ZSRC block (every LZ4 match or Snappy copy copies
// zero bytes, so the non-zero output bytes are literal bytes): the block is
// read in order as a serial decoder would, each non-zero literal byte goes
// to a sink (the apply XORs it into the receiver; the retry stream builder
// lists its unit), and each match is proven to copy zeros from a few zero
// stretches of the output so far that the library's encoder copies from.  A
// match it cannot prove, or a malformed block, stops the walk (kLStop): the
// caller hands the frame to a kernel that checks the whole output.
//
// Block formats: "A strong baseline with the Blackwell-native DE" (LZ4 block
// format; Snappy, footnote 4).  Included inside the kernel files'
// namespaces (needs kFull).

// 16 bytes through the non-coherent path, asking L2 for the 256-byte
// stretch around them (the walk reads on in order)
__device__ __forceinline__ uint4 ld_nc16_run(const uint8_t* p)
{
    uint4 v;
    asm("ld.global.nc.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p));
    return v;
}

// The body, read in order: the next bytes sit in a 64-bit register (the
// byte at the read position lowest, at least 5 of them until the body's
// last block), refilled a 32-bit word at a time from two 16-byte blocks,
// the second one in flight.  Words past the body's last block are never
// loaded (what they hold is never taken: the walks check every read against
// the body length first).
struct LaneRd {
    const uint8_t* b;
    uint32_t nblk;   // 16-byte blocks of the body (the frame is padded to 16)
    uint32_t blk;    // block in w0
    uint32_t wp;     // body offset of the next word to append
    uint32_t qn;     // bytes held in q
    uint4 w0, w1;    // blocks blk, blk + 1
    uint64_t q;
    __device__ __forceinline__ void append()
    {
        const uint32_t k = wp >> 4;
        if (k != blk) {   // k == blk + 1: words are appended in order
            w0 = w1;
            blk = k;
            if (k + 1 < nblk) w1 = ld_nc16_run(b + 16ull * (k + 1));
        }
        const uint32_t s = (wp >> 2) & 3u;
        const uint32_t w = s == 0 ? w0.x : s == 1 ? w0.y : s == 2 ? w0.z : w0.w;
        q |= uint64_t(w) << (8 * qn);
        qn += 4;
        wp += 4;
    }
    __device__ __forceinline__ void fill()
    {
        if (qn <= 4) {
            append();
            if (qn <= 4) append();
        }
    }
    __device__ __forceinline__ void init(const uint8_t* body, uint32_t n)
    {
        b = body;
        nblk = (n + 15) >> 4;
        blk = 0;
        wp = 0;
        qn = 0;
        q = 0;
        w0 = nblk > 0 ? ld_nc16_run(b) : make_uint4(0, 0, 0, 0);
        w1 = nblk > 1 ? ld_nc16_run(b + 16) : make_uint4(0, 0, 0, 0);
        fill();
    }
    // the next four bytes (the next byte lowest)
    __device__ __forceinline__ uint32_t peek() const { return uint32_t(q); }
    // move past k <= 4 bytes
    __device__ __forceinline__ void take(uint32_t k)
    {
        q >>= 8 * k;
        qn -= k;
        fill();
    }
    __device__ __forceinline__ uint32_t byte()
    {
        const uint32_t v = uint32_t(q) & 0xFFu;
        take(1);
        return v;
    }
};

// What a walk knows of the output: op bytes so far, zero from z1 on and in
// [g0, g1); the literal bytes below `done` have been XORed.  Also the zero
// stretch before each non-zero byte (its "gap"), counted in groups of 32
// non-zero bytes: the longest gap of the current group (cur) and of all
// earlier groups (best), as length << 16 | start (both below 2^16).
struct LaneOut {
    uint32_t op, z1, g0, g1, done, ev, cur, best;
};

// One literal run of ll bytes, its non-zero bytes handed to the sink
// (K.lit(output position, byte)).  kUndo: again the bytes below upto (the
// first walk's `done`), nothing else.
//
// The gaps follow the library's encoder: it copies a zero run from the
// longest gap of the earlier groups of 32 non-zero bytes, from the gap just
// before (Snappy), or from a zero it keeps as a literal (offset 1); each of
// those sources is one of the stretches kept here.
template <bool kUndo, class Sink>
__device__ __forceinline__ void lane_literals(LaneRd& R, Sink& K, LaneOut& O, uint32_t ll, uint32_t upto)
{
    // four bytes at a time; within them only the non-zero ones cost work
    for (uint32_t q = 0; q < ll; q += 4) {
        const uint32_t k = ll - q < 4 ? ll - q : 4u;
        uint32_t v = R.peek();
        if (k < 4) v &= (1u << (8 * k)) - 1;
        R.take(k);
        while (v) {
            const uint32_t j = uint32_t(__ffs(v) - 1) >> 3;
            const uint32_t b = (v >> (8 * j)) & 0xFFu;
            v &= ~(0xFFu << (8 * j));
            const uint32_t x = O.op + q + j;
            if (kUndo && x >= upto) {   // the replay is done: the step returns next
                O.op += ll;
                return;
            }
            if (!kUndo) {
                const uint32_t gap = ((x - O.z1) << 16) | O.z1;
                if (gap > O.cur) O.cur = gap;
                if ((++O.ev & 31u) == 0) {
                    if (O.cur > O.best) O.best = O.cur;
                    O.cur = 0;
                }
                O.g0 = O.z1;
                O.g1 = x;
                O.z1 = x + 1;
            }
            K.lit(x, b);
        }
    }
    O.op += ll;
    if (!kUndo) O.done = O.op;
}

// A match of ml bytes from off back at output O.op: 1 if it is in bounds and
// provably copies zeros.
__device__ __forceinline__ bool lane_match(const LaneOut& O, uint32_t off, uint32_t ml, uint32_t raw)
{
    if (off == 0 || off > O.op || ml > raw - O.op) return false;
    const uint32_t s0 = O.op - off, e0 = s0 + (ml < off ? ml : off);
    const uint32_t bs = O.best & 0xFFFFu, be = bs + (O.best >> 16);
    const uint32_t cs = O.cur & 0xFFFFu, ce = cs + (O.cur >> 16);
    return s0 >= O.z1 || (s0 >= O.g0 && e0 <= O.g1) || (s0 >= bs && e0 <= be) || (s0 >= cs && e0 <= ce);
}

// A walk's state: the body reader, the sink of the non-zero literal bytes,
// what is known of the output, the next body byte.  The caller sets up K.
template <class Sink>
struct LaneWalk {
    LaneRd R;
    Sink K;
    LaneOut O;
    uint32_t ip, n, raw, upto;
    bool sn;   // Snappy (else LZ4)
    __device__ __forceinline__ void init(bool snappy, const uint8_t* body, uint32_t bl, uint32_t raw_len,
                                         uint32_t undo_to)
    {
        R.init(body, bl);
        O = LaneOut{0, 0, 0, 0, 0, 0, 0, 0};
        ip = 0;
        n = bl;
        raw = raw_len;
        upto = undo_to;
        sn = snappy;
    }
};

// What one step of a walk found.
enum LaneStep : int { kLGo = 0, kLValid = 1, kLStop = 2 };

// An LZ4 length's extra bytes (255 continues, anything else ends it), added
// to *len, up to four at a time; false if they run past the body.
template <class W_>
__device__ __forceinline__ bool lane_len_bytes(W_& W, uint32_t* len)
{
    if (W.ip >= W.n) return false;
    const uint32_t b0 = W.R.peek() & 0xFFu;
    if (b0 != 255) {   // one byte: the common case
        *len += b0;
        ++W.ip;
        W.R.take(1);
        return true;
    }
    for (;;) {
        if (W.ip >= W.n) return false;
        const uint32_t v = W.R.peek();
        const uint32_t ff = __vcmpeq4(v, 0xFFFFFFFFu);   // 0xFF for each byte of 255
        const uint32_t avail = W.n - W.ip;
        if (ff == 0xFFFFFFFFu) {
            if (avail < 5) return false;   // the length needs a byte after these
            *len += 4 * 255;
            W.ip += 4;
            W.R.take(4);
            continue;
        }
        const uint32_t k = uint32_t(__ffs(~ff) - 1) >> 3;   // the first byte that is not 255
        if (k >= avail) return false;
        *len += 255 * k + ((v >> (8 * k)) & 0xFFu);
        W.ip += k + 1;
        W.R.take(k + 1);
        return true;
    }
}

// One LZ4 sequence (the same block format as the other walks).  kLStop: the
// block is malformed or a match is not proven to copy zeros, or (kUndo) the
// replay has reached `upto`.
template <bool kUndo, class Sink>
__device__ __forceinline__ int lz4_step(LaneWalk<Sink>& W)
{
    if (kUndo && W.O.op >= W.upto) return kLStop;
    if (W.ip >= W.n) return kLStop;
    const uint32_t tok = W.R.byte();
    ++W.ip;
    uint32_t ll = tok >> 4;
    if (ll == 15 && !lane_len_bytes(W, &ll)) return kLStop;
    if (ll > W.n - W.ip || ll > W.raw - W.O.op) return kLStop;
    lane_literals<kUndo>(W.R, W.K, W.O, ll, W.upto);
    W.ip += ll;
    if (W.ip == W.n) return W.O.op == W.raw ? kLValid : kLStop;
    if (kUndo && W.O.op >= W.upto) return kLStop;
    if (W.n - W.ip < 2) return kLStop;
    const uint32_t off = W.R.peek() & 0xFFFFu;
    W.R.take(2);
    W.ip += 2;
    uint32_t ml = tok & 15u;
    if (ml == 15 && !lane_len_bytes(W, &ml)) return kLStop;
    ml += 4;
    if (!kUndo && !lane_match(W.O, off, ml, W.raw)) return kLStop;
    W.O.op += ml;
    return kLGo;
}

// The Snappy preamble: the output length as a varint, equal to raw.
template <class Sink>
__device__ __forceinline__ bool snappy_pre(LaneWalk<Sink>& W)
{
    uint64_t v = 0;
    for (uint32_t shift = 0; shift <= 28 && W.ip < W.n; shift += 7) {
        const uint32_t b = W.R.byte();
        ++W.ip;
        v |= uint64_t(b & 127u) << shift;
        if (!(b & 128u)) return v == W.raw;
    }
    return false;
}

// One Snappy element: a literal run (1..4 length bytes past 60) or a copy.
template <bool kUndo, class Sink>
__device__ __forceinline__ int snappy_step(LaneWalk<Sink>& W)
{
    if (W.ip == W.n) return W.O.op == W.raw ? kLValid : kLStop;
    if (kUndo && W.O.op >= W.upto) return kLStop;
    const uint32_t tag = W.R.byte(), t = tag & 3u;
    ++W.ip;
    if (t == 0) {
        uint32_t len = (tag >> 2) + 1;
        if ((tag >> 2) >= 60) {
            const uint32_t nb = (tag >> 2) - 59;
            if (nb > W.n - W.ip) return kLStop;
            const uint32_t L = W.R.peek() & (nb == 4 ? 0xFFFFFFFFu : (1u << (8 * nb)) - 1);
            W.R.take(nb);
            W.ip += nb;
            if (L >= W.raw) return kLStop;
            len = L + 1;
        }
        if (len > W.n - W.ip || len > W.raw - W.O.op) return kLStop;
        lane_literals<kUndo>(W.R, W.K, W.O, len, W.upto);
        W.ip += len;
        return kLGo;
    }
    uint32_t len, off;
    if (t == 1) {
        if (W.ip >= W.n) return kLStop;
        len = ((tag >> 2) & 7u) + 4;
        off = ((tag >> 5) << 8) | W.R.byte();
        ++W.ip;
    } else {
        const uint32_t nb = t == 2 ? 2u : 4u;
        if (nb > W.n - W.ip) return kLStop;
        len = (tag >> 2) + 1;
        off = W.R.peek() & (nb == 4 ? 0xFFFFFFFFu : 0xFFFFu);
        W.R.take(nb);
        W.ip += nb;
    }
    if (!kUndo && !lane_match(W.O, off, len, W.raw)) return kLStop;
    W.O.op += len;
    return kLGo;
}

// The warp's lanes step their walks together, one sequence or element per
// lane per round, so that the warp runs converged between rounds.
template <bool kUndo, class Sink>
__device__ __forceinline__ void lane_run(LaneWalk<Sink>& W, bool act, int& res)
{
    while (__any_sync(kFull, act)) {
        if (act) {
            const int r = W.sn ? snappy_step<kUndo>(W) : lz4_step<kUndo>(W);
            if (r != kLGo) {
                act = false;
                res = r;
            }
        }
    }
}

