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


def f16_workspace(M, N, K, sms=152):
    """(counter bytes, total bytes) of the binary16-code kernel's automatic
    schedule: none when it runs whole tiles in rounds (at least half the SMs'
    worth of tiles and a last round of at least a fifth of them), else the
    balanced schedule's arrival counters of the R shared tiles, then one
    piece slot per (shared tile, CTA) pair, R + G - 1 slots of 128 x bpiece
    int32."""
    bpiece, T = f16_plan(M, N)
    if T >= sms // 2 and T % sms >= sms // 5:
        return 0, 0
    G, W, R = balanced(T, cdiv(K, 64), 16, sms)
    if R == 0 or G == R:
        return 0, 0
    cb = (R * 4 + 255) & ~255
    return cb, cb + (R + G - 1) * 128 * bpiece * 4
