// Full decoders of one LZ4 or Snappy block, run by one warp: every lane walks
// the same tokens (the reads are uniform) and the literal and match copies
// are spread over the lanes; the output goes to out[0, raw) (shared or global
// memory of the caller).  They follow the block formats as the oracle's
// strict decoders do: a block is rejected on truncation, an offset of zero
// or past the output, an overrun or an under-run of raw bytes, and, with zs
// (the frame's ZSRC flag), on a match or copy that copies a non-zero byte.
// Included inside the kernel files' namespaces (needs kFull).

// A match (LZ4) or copy (Snappy) of len bytes from off bytes back, with
// forward copy semantics (the output repeats with period off), by the whole
// warp; false (every lane) if zs and a copied byte is non-zero.  The two
// shapes the library's encoder writes get a path of their own: sources that
// do not overlap the destination, and a repeated byte (offset 1).
__device__ __forceinline__ bool copy_match(uint8_t* out, uint32_t op, uint32_t off, uint32_t len, bool zs, int lane)
{
    bool viol = false;
    if (off >= len) {
        for (uint32_t i = lane; i < len; i += 32) {
            const uint8_t b = out[op - off + i];
            out[op + i] = b;
            viol |= b != 0;
        }
    } else if (off == 1) {
        const uint8_t b = out[op - 1];
        for (uint32_t i = lane; i < len; i += 32) out[op + i] = b;
        viol = b != 0;
    } else {
        for (uint32_t i = lane; i < len; i += 32) {
            const uint8_t b = out[op - off + (i % off)];
            out[op + i] = b;
            viol |= b != 0;
        }
    }
    __syncwarp();
    return !__any_sync(kFull, zs && viol);
}

// LZ4 block ("A strong baseline with the Blackwell-native DE": the LZ4
// block format): token, literals, 2-byte offset, match-length bytes; the
// last sequence is literals only.  True (every lane) iff valid.
__device__ __noinline__ bool warp_decode_lz4(const uint8_t* src, uint32_t n, uint8_t* out, uint32_t raw, bool zs,
                                            int lane)
{
    bool good = false;
    uint32_t ip = 0, op = 0;
    for (;;) {
        if (ip >= n) break;
        const uint32_t tok = src[ip++];
        uint32_t ll = tok >> 4;
        bool ok = true;
        if (ll == 15) {
            for (;;) {
                if (ip >= n) { ok = false; break; }
                uint32_t b = src[ip++];
                ll += b;
                if (b != 255) break;
            }
        }
        if (!ok || ll > n - ip || ll > raw - op) break;
        for (uint32_t i = lane; i < ll; i += 32) out[op + i] = src[ip + i];
        __syncwarp();
        ip += ll;
        op += ll;
        if (ip == n) { good = op == raw; break; }
        if (n - ip < 2) break;
        const uint32_t off = uint32_t(src[ip]) | (uint32_t(src[ip + 1]) << 8);
        ip += 2;
        if (off == 0 || off > op) break;
        uint32_t ml = tok & 15u;
        if (ml == 15) {
            for (;;) {
                if (ip >= n) { ok = false; break; }
                uint32_t b = src[ip++];
                ml += b;
                if (b != 255) break;
            }
        }
        ml += 4;
        if (!ok || ml > raw - op) break;
        // forward copy semantics: the output repeats with period off
        if (!copy_match(out, op, off, ml, zs, lane)) break;
        op += ml;
    }
    return good;
}

// Snappy block (the same section, footnote 4): a varint of the output
// length, then literal and copy elements (copies of 1..64 bytes).
__device__ __noinline__ bool warp_decode_snappy(const uint8_t* src, uint32_t n, uint8_t* out, uint32_t raw, bool zs,
                                               int lane)
{
    bool good = false;
    uint32_t ip = 0, op = 0;
    uint64_t v = 0;
    bool pre = false;
    for (uint32_t shift = 0; shift <= 28 && ip < n; shift += 7) {
        const uint64_t b = src[ip++];
        v |= (b & 127u) << shift;
        if (!(b & 128u)) {
            pre = true;
            break;
        }
    }
    bool ok = pre && v == raw;
    while (ok && ip < n) {
        const uint32_t tag = src[ip++];
        uint32_t len, off;
        if ((tag & 3u) == 0) {
            len = (tag >> 2) + 1;
            if ((tag >> 2) >= 60) {
                const uint32_t nb = (tag >> 2) - 59;
                if (nb > n - ip) { ok = false; break; }
                len = 0;
                for (uint32_t i = 0; i < nb; ++i) len |= uint32_t(src[ip + i]) << (8 * i);
                len += 1;   // at most 2^32: wraps to 0 only for a 4-byte length, rejected below
                ip += nb;
            }
            if (len == 0 || len > n - ip || len > raw - op) { ok = false; break; }
            for (uint32_t i = lane; i < len; i += 32) out[op + i] = src[ip + i];
            __syncwarp();
            ip += len;
            op += len;
            continue;
        }
        if ((tag & 3u) == 1) {
            if (ip >= n) { ok = false; break; }
            len = ((tag >> 2) & 7u) + 4;
            off = ((tag >> 5) << 8) | src[ip++];
        } else {
            const uint32_t nb = (tag & 3u) == 2 ? 2u : 4u;
            if (nb > n - ip) { ok = false; break; }
            len = (tag >> 2) + 1;
            off = 0;
            for (uint32_t i = 0; i < nb; ++i) off |= uint32_t(src[ip + i]) << (8 * i);
            ip += nb;
        }
        if (off == 0 || off > op || len > raw - op) { ok = false; break; }
        // forward copy semantics: the output repeats with period off
        if (!copy_match(out, op, off, len, zs, lane)) { ok = false; break; }
        op += len;
    }
    good = ok && op == raw;
    return good;
}
