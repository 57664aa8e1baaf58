def decode_bytes_per_head_step(dk, dv):
    return 2 * dk * dv * 4 + dk * 2 * 3 + dk * 4 + 2
