"""GB300-native MoE token dispatch and combine."""
