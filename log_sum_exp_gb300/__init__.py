"""GB300-native row-wise log-sum-exp: out[b] = log sum_n exp(x[b, n])."""
