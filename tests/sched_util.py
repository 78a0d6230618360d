"""A restatement of the tensor-core kernels' balanced schedule (which tiles
are whole, which are shared, over how many CTAs) for sizing checks in the
tests; the library's own code is not used."""


def cdiv(a, b):
    return -(-a // b)


def balanced(T, S, min_units, sms=152):
    """(G, W, R): CTAs, rounds of whole tiles, tiles whose K stages are shared."""
    if T % sms == 0:
        return sms, T // sms, 0
    W, R = T // sms, T % sms
    if R * S < min_units * sms and W >= 1:
        W, R = W - 1, R + sms
    if R * S >= min_units * sms:
        return sms, W, R
    if W == 0:
        return max(R, min(sms, R * S // min_units)), 0, R
    return sms, cdiv(T, sms), 0


def f16_plan(M, N):
    """(bpiece, tiles) of the binary16-code kernel."""
    if M < 512:
        bpiece = cdiv(cdiv(M, cdiv(M, 256)), 32) * 32
        return bpiece, cdiv(N, 128) * cdiv(M, bpiece)
    return 256, cdiv(M, 128) * cdiv(N, 256)


def f16_schedule(M, N, K, sms=152):
    """The binary16-code kernel's automatic schedule: ("whole",), ("lock", W,
    R, P) or ("balanced", G, W, R).  Whole tiles in rounds when there are at
    least half the SMs' worth of tiles and the last round holds at least a
    fifth of them; else the rounds with the R remainder tiles cut into P =
    min(SMs // R, K stages // 16) K pieces when P >= 2; else the balanced
    schedule."""
    _, T = f16_plan(M, N)
    S = cdiv(K, 64)
    if T >= sms // 2 and T % sms >= sms // 5:
        return ("whole",)
    W, R = T // sms, T % sms
    P = min(sms // R, S // 16) if R else 1
    if P >= 2:
        return ("lock", W, R, P)
    G, W, R = balanced(T, S, 16, sms)
    return ("balanced", G, W, R)


def f16_workspace(M, N, K, sms=152):
    """(counter bytes, total bytes) of that schedule's workspace: arrival
    counters of the R shared tiles, then the piece slots of 128 x bpiece
    int32 -- P per remainder tile in lockstep rounds, one per (shared tile,
    CTA) pair (R + G - 1) in the balanced schedule; none for whole tiles."""
    bpiece, T = f16_plan(M, N)
    sc = f16_schedule(M, N, K, sms)
    if sc[0] == "whole":
        return 0, 0
    if sc[0] == "lock":
        _, W, R, P = sc
        cb = (R * 4 + 255) & ~255
        return cb, cb + R * P * 128 * bpiece * 4
    G, W, R = sc[1], sc[2], sc[3]
    if R == 0 or G == R:
        return 0, 0
    cb = (R * 4 + 255) & ~255
    return cb, cb + (R + G - 1) * 128 * bpiece * 4
