"""cattn: pluggable-map attention forward (Yat, s^tau, softmax) for GB300."""
